// Cache append: the key side of a decode step writes the new tokens' latent
// row and rotary key into the caches the attention then reads.
//
// Source: DeepSeek-V3.2-Exp atlas, "Query heads" page (excerpt mla-init and
// its prose): the layer owns a joint key-value down-projection wkv_a
// (dim -> 512 + 64) whose last 64 outputs are the shared rotary key, and a
// latent RMSNorm kv_norm over the first 512; the "Attention weights" page
// (excerpt mla-decode) reads kv_cache[:bsz, :end_pos] and pe_cache[:bsz,
// :end_pos].  The pages do not print the write itself; this kernel takes the
// plain reading: token s of T new tokens of sequence b sits at position
// end_pos[b] - T + s, its normalised latent goes to kv_cache[b][pos] and its
// rotary key, rotated (interleaved pairs) at pos, to pe_cache[b][pos].
//
// One CTA of 128 threads per token: each thread holds 4 latent features; the
// sum of squares is reduced across the CTA in fp32; threads 0..31 rotate one
// rotary pair each.
#include "common.cuh"

namespace mla {
namespace app {

constexpr int THREADS = 128;

__global__ void __launch_bounds__(THREADS) append_kernel(const uint16_t *__restrict__ kv_a,
                                                         const float *__restrict__ norm_w, float eps,
                                                         const float2 *__restrict__ cis, int max_seq_len,
                                                         const int32_t *__restrict__ end_pos, int T, int S_cap,
                                                         uint16_t *__restrict__ kv_cache,
                                                         uint16_t *__restrict__ pe_cache, int32_t *status) {
    __shared__ float part[THREADS / 32];
    const int tok = blockIdx.x;           // b * T + s
    const int b = tok / T, s = tok - b * T;
    const int tid = threadIdx.x;
    const int e = end_pos[b];
    if (e < T || e > S_cap) {
        if (tid == 0 && s == 0) report(status, MLA_DEV_BAD_END_POS);
        return;
    }
    const int pos = e - T + s;
    if (pos >= max_seq_len) {
        if (tid == 0) report(status, MLA_DEV_BAD_POSITION);
        return;
    }
    const uint16_t *src = kv_a + (size_t)tok * QL;
    const uint2 raw = *reinterpret_cast<const uint2 *>(src + 4 * tid);
    float x[4] = {bflo(raw.x), bfhi(raw.x), bflo(raw.y), bfhi(raw.y)};
    float ss = x[0] * x[0] + x[1] * x[1] + x[2] * x[2] + x[3] * x[3];
#pragma unroll
    for (int o = 16; o; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    if ((tid & 31) == 0) part[tid >> 5] = ss;
    __syncthreads();
    const float total = part[0] + part[1] + part[2] + part[3];
    const float inv = rsqrtf(total / float(C) + eps);
    const float4 w = *reinterpret_cast<const float4 *>(norm_w + 4 * tid);
    uint16_t *kv_row = kv_cache + ((size_t)b * S_cap + pos) * C;
    uint2 out;
    out.x = uint32_t(f2bf(x[0] * inv * w.x)) | (uint32_t(f2bf(x[1] * inv * w.y)) << 16);
    out.y = uint32_t(f2bf(x[2] * inv * w.z)) | (uint32_t(f2bf(x[3] * inv * w.w)) << 16);
    *reinterpret_cast<uint2 *>(kv_row + 4 * tid) = out;
    if (tid < NPAIR) {
        const uint32_t pr = *reinterpret_cast<const uint32_t *>(src + C + 2 * tid);
        const float x0 = bflo(pr), x1 = bfhi(pr);
        const float2 cs = cis[(size_t)pos * NPAIR + tid];
        uint16_t *pe_row = pe_cache + ((size_t)b * S_cap + pos) * DR;
        *reinterpret_cast<uint32_t *>(pe_row + 2 * tid) =
            uint32_t(f2bf(x0 * cs.x - x1 * cs.y)) | (uint32_t(f2bf(x0 * cs.y + x1 * cs.x)) << 16);
    }
}

}  // namespace app
}  // namespace mla

using namespace mla;

extern "C" int mla_cache_append(const mla_bf16 *kv_a, const float *kv_norm_w, float eps, const float *cis,
                                int max_seq_len, const int32_t *end_pos, int B, int T, mla_bf16 *kv_cache,
                                mla_bf16 *pe_cache, int S_cap, int32_t *dev_status, mla_stream_t stream) {
    if (!kv_a || !kv_norm_w || !cis || !end_pos || !kv_cache || !pe_cache) return MLA_ERR_NULL;
    if (!aligned16(kv_a) || !aligned16(kv_norm_w) || !aligned16(cis) || !aligned16(kv_cache) ||
        !aligned16(pe_cache))
        return MLA_ERR_ALIGN;
    if (B < 1 || T < 1 || (long long)B * T > (1ll << 31) - 1 || S_cap < 1 || max_seq_len < 1 || !(eps >= 0.f))
        return MLA_ERR_SIZE;
    app::append_kernel<<<B * T, app::THREADS, 0, (cudaStream_t)stream>>>(
        kv_a, kv_norm_w, eps, reinterpret_cast<const float2 *>(cis), max_seq_len, end_pos, T, S_cap, kv_cache,
        pe_cache, dev_status);
    count_launches(1);
    return cudaGetLastError() == cudaSuccess ? MLA_OK : MLA_ERR_CUDA;
}
