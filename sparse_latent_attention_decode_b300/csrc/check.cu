// mla_check_selection: flags a position that occurs twice among the valid
// entries of one selection row.
//
// Source: DeepSeek-V3.2-Exp atlas, "Attention weights" page, excerpt
// mla-decode: the mask is a row of -inf with zeros scattered in at the
// selected positions, so the selection is a set; the attention kernels add
// one term per valid entry and would count a repeated position twice.
#include "common.cuh"
#include "kernels.cuh"

namespace mla {
namespace check {

// one block per query row r = b*T + s: the positions the row can see, [0, e)
// with e = end_pos[b] - T + s + 1, are marked in a shared-memory bitmap; a
// position found already marked is a duplicate.  Padding is never marked.
__global__ void __launch_bounds__(256) check_kernel(const int32_t *__restrict__ topk, int K,
                                                    const int32_t *__restrict__ end_pos, int T, int S_cap,
                                                    int32_t *status) {
    extern __shared__ uint32_t bits[];
    const int r = blockIdx.x, b = r / T, s = r - b * T;
    const int ep = end_pos[b];
    if (ep < T || ep > S_cap) {   // the decode skips the sequence and reports it
        if (threadIdx.x == 0 && s == 0) report(status, MLA_DEV_BAD_END_POS);
        return;
    }
    const int e = ep - T + s + 1;
    for (int i = threadIdx.x; i < (e + 31) / 32; i += blockDim.x) bits[i] = 0u;
    __syncthreads();
    const int32_t *row = topk + (size_t)r * K;
    bool dup = false;
    for (int i = threadIdx.x; i < K; i += blockDim.x) {
        const int t = row[i];
        if (t < 0 || t >= e) continue;
        const uint32_t m = 1u << (t & 31);
        dup |= (atomicOr(&bits[t >> 5], m) & m) != 0u;
    }
    if (__syncthreads_or(dup) && threadIdx.x == 0) report(status, MLA_DEV_DUPLICATE_INDEX);
}

}  // namespace check
}  // namespace mla

using namespace mla;

extern "C" int mla_check_selection(const int32_t *topk_idx, int K, const int32_t *end_pos, int n_seq, int T,
                                   int S_cap, int32_t *dev_status, mla_stream_t stream) {
    if (!topk_idx || !end_pos || !dev_status) return MLA_ERR_NULL;
    if (!aligned16(topk_idx)) return MLA_ERR_ALIGN;
    if (n_seq < 1 || T < 1 || (long long)n_seq * T > 4096 || K < 1 || K > (1 << 20) || S_cap < 1 ||
        S_cap > MLA_CHECK_MAX_S_CAP)
        return MLA_ERR_SIZE;
    const int smem = (S_cap + 31) / 32 * 4;   // the bitmap of the longest visible range
    static std::atomic<bool> smem_set[64];
    if (!smem_attr_once(smem_set, check::check_kernel, (MLA_CHECK_MAX_S_CAP + 31) / 32 * 4)) return MLA_ERR_CUDA;
    check::check_kernel<<<n_seq * T, 256, smem, (cudaStream_t)stream>>>(topk_idx, K, end_pos, T, S_cap, dev_status);
    count_launches(1);
    return cudaGetLastError() == cudaSuccess ? MLA_OK : MLA_ERR_CUDA;
}
