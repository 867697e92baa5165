// Launchers shared between translation units of the library.
#pragma once

#include "common.cuh"

namespace mla {

int launch_out_up(const float *o_lat, const uint16_t *wkv_b, int B, float *out, cudaStream_t s);

}  // namespace mla
