// Value up-projection: out[b,h,d] = sum_c o[b,h,c] * W_UV[h][d][c].
//
// Source: DeepSeek-V3.2-Exp atlas, "Attention weights" page, excerpt
// mla-decode (last einsum, wkv_b[:, -v_head_dim:]).
#include "common.cuh"
#include "kernels.cuh"

namespace mla {

constexpr int UP_BT = 8;   // sequences per CTA
constexpr int UP_CK = 64;  // latent columns per smem tile

// grid (H, ceil(B/8)), 128 threads: thread = one output feature d of one head.
// o is rounded to bf16 before the product (the operands are bf16; fp32 sums).
__global__ void __launch_bounds__(128) out_up_simt_kernel(const float *__restrict__ o_lat,
                                                          const uint16_t *__restrict__ wkv_b, int B,
                                                          float *__restrict__ out) {
    __shared__ uint32_t ws[DV][UP_CK / 2 + 1];
    __shared__ float os[UP_BT][UP_CK];
    const int h = blockIdx.x, b0 = blockIdx.y * UP_BT, d = threadIdx.x;
    const int nb = min(UP_BT, B - b0);
    float acc[UP_BT];
#pragma unroll
    for (int j = 0; j < UP_BT; ++j) acc[j] = 0.f;
    const uint32_t *w_uv = reinterpret_cast<const uint32_t *>(wkv_b + ((size_t)h * WROWS + DN) * C);
    for (int c0 = 0; c0 < C; c0 += UP_CK) {
        for (int u = threadIdx.x; u < DV * UP_CK / 2; u += 128) {
            const int r = u / (UP_CK / 2), w = u % (UP_CK / 2);
            ws[r][w] = w_uv[(size_t)r * (C / 2) + c0 / 2 + w];
        }
        for (int u = threadIdx.x; u < UP_BT * UP_CK; u += 128) {
            const int j = u / UP_CK, c = u % UP_CK;
            os[j][c] = j < nb ? bf2f(f2bf(o_lat[((size_t)(b0 + j) * H + h) * C + c0 + c])) : 0.f;
        }
        __syncthreads();
        for (int w = 0; w < UP_CK / 2; ++w) {
            const uint32_t kw = ws[d][w];
            const float lo = bflo(kw), hi = bfhi(kw);
#pragma unroll
            for (int j = 0; j < UP_BT; ++j) acc[j] = fmaf(os[j][2 * w + 1], hi, fmaf(os[j][2 * w], lo, acc[j]));
        }
        __syncthreads();
    }
    for (int j = 0; j < nb; ++j) out[((size_t)(b0 + j) * H + h) * DV + d] = acc[j];
}

int launch_out_up(const float *o_lat, const uint16_t *wkv_b, int B, float *out, cudaStream_t s) {
    dim3 grid(H, (B + UP_BT - 1) / UP_BT);
    out_up_simt_kernel<<<grid, 128, 0, s>>>(o_lat, wkv_b, B, out);
    count_launches(1);
    return cudaGetLastError() == cudaSuccess ? MLA_OK : MLA_ERR_CUDA;
}

}  // namespace mla

using namespace mla;

extern "C" int mla_out_up(const float *o_lat, const mla_bf16 *wkv_b, int B, float *out, mla_stream_t stream) {
    if (!o_lat || !wkv_b || !out) return MLA_ERR_NULL;
    if (!aligned16(o_lat) || !aligned16(wkv_b) || !aligned16(out)) return MLA_ERR_ALIGN;
    if (B < 1 || B > 4096) return MLA_ERR_SIZE;
    return launch_out_up(o_lat, wkv_b, B, out, (cudaStream_t)stream);
}
