// Query of the latent attention: key absorption with the RoPE of q_pe fused in.
//
// Source: DeepSeek-V3.2-Exp atlas, "Query content heads" page, excerpt
// mla-decode (first einsum: q_nope . W_UK per head), and "Rotated query part"
// page, excerpt apply-rope (pair rotation of q_pe).
#include "common.cuh"

namespace mla {

constexpr int ABS_BT = 16;  // sequences per CTA

// grid (H, C/128, ceil(B/16)), 128 threads: thread = one latent column c of
// one head; W_UK[h][d][c] is read once per CTA, coalesced over c.
__global__ void __launch_bounds__(128) absorb_simt_kernel(
    const uint16_t *__restrict__ q_nope, const uint16_t *__restrict__ q_pe, const float2 *__restrict__ cis,
    int max_seq_len, const int32_t *__restrict__ end_pos, const uint16_t *__restrict__ wkv_b, int B,
    uint16_t *__restrict__ q_lat, int32_t *status) {
    __shared__ float qs[ABS_BT][DN];
    const int h = blockIdx.x, c = blockIdx.y * 128 + threadIdx.x, b0 = blockIdx.z * ABS_BT;
    const int nb = min(ABS_BT, B - b0);
    for (int k = threadIdx.x; k < ABS_BT * DN; k += 128) {
        const int j = k / DN, d = k % DN;
        qs[j][d] = j < nb ? bf2f(q_nope[((size_t)(b0 + j) * H + h) * DN + d]) : 0.f;
    }
    __syncthreads();
    float acc[ABS_BT];
#pragma unroll
    for (int j = 0; j < ABS_BT; ++j) acc[j] = 0.f;
    const uint16_t *w = wkv_b + (size_t)h * WROWS * C + c;
    for (int d = 0; d < DN; ++d) {
        const float wv = bf2f(w[(size_t)d * C]);
#pragma unroll
        for (int j = 0; j < ABS_BT; ++j) acc[j] = fmaf(qs[j][d], wv, acc[j]);
    }
    for (int j = 0; j < nb; ++j) q_lat[((size_t)(b0 + j) * H + h) * QL + c] = f2bf(acc[j]);

    // fused RoPE prologue: the c-chunk-0 CTA of each head rotates q_pe
    if (blockIdx.y == 0 && threadIdx.x < NPAIR) {
        const int i = threadIdx.x;
        for (int j = 0; j < nb; ++j) {
            const int b = b0 + j;
            const int pos = end_pos[b] - 1;
            uint32_t packed = 0;
            if (pos >= 0 && pos < max_seq_len) {
                const uint32_t wv = reinterpret_cast<const uint32_t *>(q_pe + ((size_t)b * H + h) * DR)[i];
                const float x0 = bflo(wv), x1 = bfhi(wv);
                const float2 cs = cis[(size_t)pos * NPAIR + i];
                packed = uint32_t(f2bf(x0 * cs.x - x1 * cs.y)) | (uint32_t(f2bf(x0 * cs.y + x1 * cs.x)) << 16);
            } else if (i == 0 && h == 0) {
                report(status, MLA_DEV_BAD_POSITION);
            }
            reinterpret_cast<uint32_t *>(q_lat + ((size_t)b * H + h) * QL + C)[i] = packed;
        }
    }
}

}  // namespace mla

using namespace mla;

extern "C" int mla_absorb_q(const mla_bf16 *q_nope, const mla_bf16 *q_pe, const float *cis, int max_seq_len,
                            const int32_t *end_pos, const mla_bf16 *wkv_b, int B, mla_bf16 *q_lat,
                            int32_t *dev_status, mla_stream_t stream) {
    if (!q_nope || !q_pe || !cis || !end_pos || !wkv_b || !q_lat) return MLA_ERR_NULL;
    if (!aligned16(q_nope) || !aligned16(q_pe) || !aligned16(cis) || !aligned16(wkv_b) || !aligned16(q_lat))
        return MLA_ERR_ALIGN;
    if (B < 1 || B > 4096 || max_seq_len < 1) return MLA_ERR_SIZE;
    dim3 grid(H, C / 128, (B + ABS_BT - 1) / ABS_BT);
    absorb_simt_kernel<<<grid, 128, 0, (cudaStream_t)stream>>>(q_nope, q_pe, reinterpret_cast<const float2 *>(cis),
                                                              max_seq_len, end_pos, wkv_b, B, q_lat, dev_status);
    count_launches(1);
    return cudaGetLastError() == cudaSuccess ? MLA_OK : MLA_ERR_CUDA;
}
