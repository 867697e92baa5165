// Block-scaled fp8 (e4m3) weight -> bf16: the dequantisation the attention
// takes its wkv_b through when the checkpoint stores it in fp8.
//
// Source: DeepSeek-V3.2-Exp atlas, "Rotated query part" / "Query content
// heads" pages, excerpt mla-decode: on first use the layer calls
// weight_dequant(wkv_b.weight, wkv_b.scale) and keeps the result as the wkv_b
// of the absorbed path.  The pages name the call but not the scale format;
// this library reads it as one fp32 multiplier per block x block tile of the
// weight (the scale grid [ceil(rows/block)][ceil(cols/block)], row-major) and
// takes the product in fp32 before rounding it to bf16 (round to nearest even).
//
// The kernel is a pure stream: 1 byte in and 2 bytes out per element, plus one
// scale per tile that stays in L1/L2.  Each thread turns 16 codes (one 16-byte
// load) into 16 bf16 values (two 16-byte stores); the grid strides over the
// matrix with a whole number of CTAs per SM.
#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include "common.cuh"

namespace mla {
namespace dq {

__device__ __forceinline__ float2 e4m3x2_to_f2(uint16_t two) {
    const __half2_raw h = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(two), __NV_E4M3);
    return __half22float2(*reinterpret_cast<const __half2 *>(&h));
}

__device__ __forceinline__ uint32_t pack_bf2(float lo, float hi) {
    const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<const uint32_t *>(&v);
}

// 16 consecutive elements of one row share a scale (cols % 16 == 0 and
// block % 16 == 0), so one thread handles them with vector loads and stores.
__global__ void __launch_bounds__(256) dequant_vec_kernel(const uint4 *__restrict__ w, const float *__restrict__ scale,
                                                          int cols, int block, int scale_cols, long long n16,
                                                          uint4 *__restrict__ out) {
    const int chunks_per_row = cols / 16;
    for (long long k = blockIdx.x * (long long)blockDim.x + threadIdx.x; k < n16;
         k += (long long)gridDim.x * blockDim.x) {
        const long long r = k / chunks_per_row;
        const int c = int(k - r * chunks_per_row) * 16;
        const float s = __ldg(scale + (r / block) * scale_cols + c / block);
        const uint4 q = __ldcs(w + k);
        const uint32_t words[4] = {q.x, q.y, q.z, q.w};
        uint32_t o[8];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const float2 a = e4m3x2_to_f2(uint16_t(words[j] & 0xffffu));
            const float2 b = e4m3x2_to_f2(uint16_t(words[j] >> 16));
            o[2 * j] = pack_bf2(__fmul_rn(a.x, s), __fmul_rn(a.y, s));
            o[2 * j + 1] = pack_bf2(__fmul_rn(b.x, s), __fmul_rn(b.y, s));
        }
        __stcs(out + 2 * k, make_uint4(o[0], o[1], o[2], o[3]));
        __stcs(out + 2 * k + 1, make_uint4(o[4], o[5], o[6], o[7]));
    }
}

// Any shape, any block size: one element per thread and iteration.
__global__ void __launch_bounds__(256) dequant_any_kernel(const uint8_t *__restrict__ w, const float *__restrict__ scale,
                                                          int cols, int block, int scale_cols, long long n,
                                                          uint16_t *__restrict__ out) {
    for (long long k = blockIdx.x * (long long)blockDim.x + threadIdx.x; k < n;
         k += (long long)gridDim.x * blockDim.x) {
        const long long r = k / cols;
        const int c = int(k - r * cols);
        const float s = __ldg(scale + (r / block) * scale_cols + c / block);
        const float2 v = e4m3x2_to_f2(uint16_t(w[k]));
        out[k] = f2bf(__fmul_rn(v.x, s));
    }
}

}  // namespace dq
}  // namespace mla

using namespace mla;

extern "C" int mla_weight_dequant_fp8(const uint8_t *w, const float *scale, int rows, int cols, int block,
                                      mla_bf16 *out, mla_stream_t stream) {
    if (!w || !scale || !out) return MLA_ERR_NULL;
    if (rows < 1 || cols < 1 || block < 1 || (long long)rows * cols > (1ll << 40)) return MLA_ERR_SIZE;
    if ((reinterpret_cast<uintptr_t>(scale) & 3u) != 0 || (reinterpret_cast<uintptr_t>(out) & 1u) != 0)
        return MLA_ERR_ALIGN;
    int dev = 0, sms = 148;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return MLA_ERR_CUDA;
    const int scale_cols = (cols + block - 1) / block;
    const long long n = (long long)rows * cols;
    const int threads = 256;
    const bool vec = cols % 16 == 0 && block % 16 == 0 && aligned16(w) && aligned16(out);
    const long long work = vec ? n / 16 : n;
    const long long want = (work + threads - 1) / threads;
    // 8 CTAs of 256 threads fill an SM; beyond that the grid strides
    const long long cap = (long long)sms * 8;
    const int blocks = int(want < cap ? want : cap);
    if (vec)
        dq::dequant_vec_kernel<<<blocks, threads, 0, (cudaStream_t)stream>>>(
            reinterpret_cast<const uint4 *>(w), scale, cols, block, scale_cols, work, reinterpret_cast<uint4 *>(out));
    else
        dq::dequant_any_kernel<<<blocks, threads, 0, (cudaStream_t)stream>>>(w, scale, cols, block, scale_cols, n,
                                                                             out);
    count_launches(1);
    return cudaGetLastError() == cudaSuccess ? MLA_OK : MLA_ERR_CUDA;
}
