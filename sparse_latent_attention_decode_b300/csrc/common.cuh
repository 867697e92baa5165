// Shared device helpers of the sparse MLA decode library.
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "mla_decode.h"

namespace mla {

constexpr int H = MLA_N_HEADS;       // 128 heads
constexpr int DN = MLA_D_NOPE;       // 128 content features per head
constexpr int DR = MLA_D_ROPE;       // 64 rotary features
constexpr int DV = MLA_D_V;          // 128 value features per head
constexpr int C = MLA_KV_LORA;       // 512 latent features
constexpr int QL = MLA_Q_LAT;        // 576 = C + DR
constexpr int NPAIR = DR / 2;        // 32 rotary pairs
constexpr int WROWS = DN + DV;       // 256 rows of wkv_b per head

__device__ __forceinline__ float bf2f(uint16_t v) { return __uint_as_float(uint32_t(v) << 16); }
__device__ __forceinline__ uint16_t f2bf(float f) {
    return __bfloat16_as_ushort(__float2bfloat16_rn(f));
}
__device__ __forceinline__ float bflo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bfhi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

__device__ __forceinline__ void report(int32_t *status, int bits) {
    if (status) atomicOr(reinterpret_cast<int *>(status), bits);
}

// per-thread profiling hook (see mla_profile_hook)
struct ProfileHook {
    cudaEvent_t start = nullptr, stop = nullptr;
    int64_t *launches = nullptr;
};
ProfileHook &profile_hook();
inline void count_launches(int n) {
    if (profile_hook().launches) *profile_hook().launches += n;
}

inline bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Limit of the bounded on-chip waits of the kernels that drain their own
// in-flight copies and MMAs before they give up (see mla_set_wait_limit_ns);
// read at launch and passed to the kernel.
uint64_t wait_limit_ns();
// Every kernel that gives up a wait first waits, for at most this long, for
// the copies and MMAs it has already issued, so that nothing it started
// still writes its shared memory or tensor memory after it has released them.
constexpr uint64_t DRAIN_NS = 1000000000ull;

}  // namespace mla
