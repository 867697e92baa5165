// Launchers and host helpers shared between translation units of the library.
#pragma once

#include <cuda.h>

#include "common.cuh"

namespace mla {

int launch_out_up(const float *o_lat, const uint16_t *wkv_b, int B, float *out, int32_t *status, cudaStream_t s);

// Sparse attention (tensor-core kernel + split combine).  Writes the
// normalised latent output o [B][128][512] fp32 to o_out.  ws must hold
// attn_workspace(B, K) bytes (256-byte aligned).
size_t attn_workspace(int B, int K, int *n_split = nullptr, int *split_len = nullptr);
int launch_attn(const uint16_t *q_lat, const uint16_t *kv, const uint16_t *pe, int S_cap, const int32_t *topk, int K,
                const int32_t *end_pos, int B, float softmax_scale, float *o_out, void *ws, int32_t *status,
                cudaStream_t s, int *launches);

// TMA tensor map of a bf16 tensor (dims[0] innermost); false on failure.
bool make_tmap_bf16(CUtensorMap *map, const void *base, int rank, const uint64_t *dims,
                    const uint64_t *strides_bytes, const uint32_t *box, CUtensorMapSwizzle swizzle);

}  // namespace mla
