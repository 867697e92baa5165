// Sparse latent attention over the selected cache rows: scores, softmax over
// the selected set (online, split over blocks of the selection), PV, split
// combine, and the optional value up-projection.
//
// Source: DeepSeek-V3.2-Exp atlas, "Attention weights" page, excerpt
// mla-decode: scores = (q~ . kv + q_pe . pe) * scale, + selection mask,
// softmax over keys, probabilities . kv, then . W_UV.
#include "common.cuh"
#include "kernels.cuh"

#include <math.h>

namespace mla {

constexpr int DK_KB = 32;       // selected rows per block
constexpr int DK_HG = 16;       // heads per CTA
constexpr int DK_SPLIT = 256;   // selection entries per split
constexpr int DK_ROWW = QL / 2 + 1;  // 32-bit words per smem row (+1 pad: conflict-free)

struct DecodeSmem {
    float q[DK_HG][QL];
    uint32_t k[DK_KB][DK_ROWW];
    float p[DK_HG][DK_KB];
    float fac[DK_HG], m[DK_HG], l[DK_HG];
    int idx[DK_KB];
};

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// grid (nsplit, B, H/16), 256 threads.  Writes, per (sequence, split, head),
// the unnormalised partial o (fp32 [512]) and its (running max, sum).
__global__ void __launch_bounds__(256) decode_simt_kernel(
    const uint16_t *__restrict__ q_lat, const uint16_t *__restrict__ kv, const uint16_t *__restrict__ pe, int S_cap,
    const int32_t *__restrict__ topk, int K, const int32_t *__restrict__ end_pos, float scale,
    float *__restrict__ part_o, float2 *__restrict__ part_ml, int nsplit, int32_t *status) {
    extern __shared__ __align__(16) unsigned char smem_raw[];
    DecodeSmem &sm = *reinterpret_cast<DecodeSmem *>(smem_raw);
    const int s = blockIdx.x, b = blockIdx.y, g = blockIdx.z, tid = threadIdx.x;
    const int lane = tid & 31, warp = tid >> 5;
    const int e = end_pos[b];
    const size_t part_row = ((size_t)b * nsplit + s) * H + g * DK_HG;
    const int hh = tid >> 4, cw = tid & 15;  // PV: head within group, column word lane

    float o[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) o[i] = 0.f;

    if (e < 1 || e > S_cap) {
        if (s == 0 && g == 0 && tid == 0) report(status, MLA_DEV_BAD_END_POS);
        if (tid < DK_HG) sm.m[tid] = -INFINITY, sm.l[tid] = 0.f;
    } else {
        for (int u = tid; u < DK_HG * QL; u += 256) {
            const int j = u / QL, c = u % QL;
            sm.q[j][c] = bf2f(q_lat[((size_t)b * H + g * DK_HG + j) * QL + c]);
        }
        if (tid < DK_HG) sm.m[tid] = -INFINITY, sm.l[tid] = 0.f;
        const int t0 = s * DK_SPLIT, t1 = min(K, t0 + DK_SPLIT);
        for (int kb = t0; kb < t1; kb += DK_KB) {
            const int nk = min(DK_KB, t1 - kb);
            __syncthreads();
            if (tid < DK_KB) {
                int id = tid < nk ? topk[(size_t)b * K + kb + tid] : -1;
                sm.idx[tid] = (id >= 0 && id < e) ? id : -1;
            }
            __syncthreads();
            // gather the selected rows: 72 16-byte chunks per row (64 latent + 8 rotary)
            for (int u = tid; u < DK_KB * 72; u += 256) {
                const int j = u / 72, q16 = u % 72;
                const int id = sm.idx[j];
                uint4 v = make_uint4(0, 0, 0, 0);
                if (id >= 0) {
                    if (q16 < 64)
                        v = reinterpret_cast<const uint4 *>(kv + ((size_t)b * S_cap + id) * C)[q16];
                    else
                        v = reinterpret_cast<const uint4 *>(pe + ((size_t)b * S_cap + id) * DR)[q16 - 64];
                }
                uint32_t *dst = &sm.k[j][q16 * 4];
                dst[0] = v.x, dst[1] = v.y, dst[2] = v.z, dst[3] = v.w;
            }
            __syncthreads();
            {  // scores: lane = row, warp = heads (warp, warp+8)
                const int j = lane, h0 = warp, h1 = warp + 8;
                float a0 = 0.f, a1 = 0.f;
                for (int w = 0; w < QL / 2; ++w) {
                    const uint32_t kw = sm.k[j][w];
                    const float k0 = bflo(kw), k1 = bfhi(kw);
                    a0 = fmaf(sm.q[h0][2 * w + 1], k1, fmaf(sm.q[h0][2 * w], k0, a0));
                    a1 = fmaf(sm.q[h1][2 * w + 1], k1, fmaf(sm.q[h1][2 * w], k0, a1));
                }
                const bool ok = sm.idx[j] >= 0;
                sm.p[h0][j] = ok ? a0 * scale : -INFINITY;
                sm.p[h1][j] = ok ? a1 * scale : -INFINITY;
            }
            __syncthreads();
            // online softmax update, one warp per head pair
#pragma unroll
            for (int r = 0; r < 2; ++r) {
                const int h = warp + 8 * r;
                const float sc = sm.p[h][lane];
                const float m_old = sm.m[h];
                const float m_new = fmaxf(m_old, warp_max(sc));
                float p = 0.f, f = 1.f;
                if (m_new != -INFINITY) {
                    p = (sc == -INFINITY) ? 0.f : expf(sc - m_new);
                    f = (m_old == -INFINITY) ? 0.f : expf(m_old - m_new);
                }
                const float tot = warp_sum(p);
                sm.p[h][lane] = p;
                __syncwarp();
                if (lane == 0) {
                    sm.l[h] = sm.l[h] * f + tot;
                    sm.m[h] = m_new;
                    sm.fac[h] = f;
                }
            }
            __syncthreads();
            {  // PV: thread owns head hh, latent words cw + 16 i
                const float f = sm.fac[hh];
#pragma unroll
                for (int i = 0; i < 32; ++i) o[i] *= f;
                for (int j = 0; j < nk; ++j) {
                    const float p = sm.p[hh][j];
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        const uint32_t kw = sm.k[j][cw + 16 * i];
                        o[2 * i] = fmaf(p, bflo(kw), o[2 * i]);
                        o[2 * i + 1] = fmaf(p, bfhi(kw), o[2 * i + 1]);
                    }
                }
            }
        }
    }
    __syncthreads();
    float *dst = part_o + (part_row + hh) * C;
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        const int w = cw + 16 * i;
        dst[2 * w] = o[2 * i];
        dst[2 * w + 1] = o[2 * i + 1];
    }
    if (tid < DK_HG) part_ml[part_row + tid] = make_float2(sm.m[tid], sm.l[tid]);
}

// grid (B, H), 128 threads x 4 columns: merge the splits of one (sequence,
// head) by their running maxima and normalise.  Nothing selected -> zeros.
__global__ void __launch_bounds__(128) combine_kernel(const float *__restrict__ part_o,
                                                      const float2 *__restrict__ part_ml, int nsplit,
                                                      float *__restrict__ o_lat) {
    const int b = blockIdx.x, h = blockIdx.y, c = threadIdx.x * 4;
    float M = -INFINITY;
    for (int s = 0; s < nsplit; ++s) M = fmaxf(M, part_ml[((size_t)b * nsplit + s) * H + h].x);
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    float L = 0.f;
    if (M != -INFINITY) {
        for (int s = 0; s < nsplit; ++s) {
            const size_t row = ((size_t)b * nsplit + s) * H + h;
            const float2 ml = part_ml[row];
            if (ml.x == -INFINITY) continue;
            const float w = expf(ml.x - M);
            L = fmaf(w, ml.y, L);
            const float4 v = *reinterpret_cast<const float4 *>(part_o + row * C + c);
            acc.x = fmaf(w, v.x, acc.x), acc.y = fmaf(w, v.y, acc.y);
            acc.z = fmaf(w, v.z, acc.z), acc.w = fmaf(w, v.w, acc.w);
        }
    }
    const float inv = L > 0.f ? 1.f / L : 0.f;
    *reinterpret_cast<float4 *>(o_lat + ((size_t)b * H + h) * C + c) =
        make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
}

struct WsLayout {
    size_t part_o, part_ml, o_lat, total;
    int nsplit;
};

static inline size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

static WsLayout ws_layout(int B, int K) {
    WsLayout w{};
    w.nsplit = (K + DK_SPLIT - 1) / DK_SPLIT;
    const size_t rows = (size_t)B * w.nsplit * H;
    w.part_o = 0;
    w.part_ml = align256(rows * C * sizeof(float));
    w.o_lat = w.part_ml + align256(rows * sizeof(float2));
    w.total = w.o_lat + align256((size_t)B * H * C * sizeof(float));
    return w;
}

}  // namespace mla

using namespace mla;

extern "C" size_t mla_sparse_decode_workspace_size(int B, int K) {
    if (B < 1 || B > 4096 || K < 1 || K > (1 << 20)) return 0;
    return ws_layout(B, K).total;
}

extern "C" int mla_sparse_decode(const mla_bf16 *q_lat, const mla_bf16 *kv_cache, const mla_bf16 *pe_cache,
                                 int S_cap, const int32_t *topk_idx, int K, const int32_t *end_pos, int B,
                                 float softmax_scale, const mla_bf16 *wkv_b, float *out, void *workspace,
                                 size_t ws_bytes, int32_t *dev_status, mla_stream_t stream) {
    if (!q_lat || !kv_cache || !pe_cache || !topk_idx || !end_pos || !out || !workspace) return MLA_ERR_NULL;
    if (!aligned16(q_lat) || !aligned16(kv_cache) || !aligned16(pe_cache) || !aligned16(topk_idx) ||
        !aligned16(out) || (wkv_b && !aligned16(wkv_b)) || (reinterpret_cast<uintptr_t>(workspace) & 255u))
        return MLA_ERR_ALIGN;
    if (B < 1 || B > 4096 || K < 1 || K > (1 << 20) || S_cap < 1) return MLA_ERR_SIZE;
    const WsLayout L = ws_layout(B, K);
    if (ws_bytes < L.total) return MLA_ERR_WORKSPACE;
    cudaStream_t s = (cudaStream_t)stream;
    char *ws = static_cast<char *>(workspace);
    float *part_o = reinterpret_cast<float *>(ws + L.part_o);
    float2 *part_ml = reinterpret_cast<float2 *>(ws + L.part_ml);
    float *o_lat = wkv_b ? reinterpret_cast<float *>(ws + L.o_lat) : out;

    const int smem = int(sizeof(DecodeSmem));
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return MLA_ERR_CUDA;
    static bool attr_set[64] = {};
    if (dev < 0 || dev >= 64 || !attr_set[dev]) {
        if (cudaFuncSetAttribute(decode_simt_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) !=
            cudaSuccess)
            return MLA_ERR_CUDA;
        if (dev >= 0 && dev < 64) attr_set[dev] = true;
    }
    dim3 grid(L.nsplit, B, H / DK_HG);
    const ProfileHook &hook = profile_hook();
    const bool timed = hook.start && hook.stop;
    if (timed && cudaEventRecord(hook.start, s) != cudaSuccess) return MLA_ERR_CUDA;
    decode_simt_kernel<<<grid, 256, smem, s>>>(q_lat, kv_cache, pe_cache, S_cap, topk_idx, K, end_pos,
                                               softmax_scale, part_o, part_ml, L.nsplit, dev_status);
    if (cudaGetLastError() != cudaSuccess) return MLA_ERR_CUDA;
    if (timed && cudaEventRecord(hook.stop, s) != cudaSuccess) return MLA_ERR_CUDA;
    combine_kernel<<<dim3(B, H), 128, 0, s>>>(part_o, part_ml, L.nsplit, o_lat);
    if (cudaGetLastError() != cudaSuccess) return MLA_ERR_CUDA;
    count_launches(2);
    if (wkv_b) return launch_out_up(o_lat, wkv_b, B, out, s);
    return MLA_OK;
}

extern "C" const char *mla_status_string(int code) {
    switch (code) {
        case MLA_OK: return "ok";
        case MLA_ERR_NULL: return "a required pointer is NULL";
        case MLA_ERR_ALIGN: return "a pointer is not 16-byte aligned (workspace: 256-byte)";
        case MLA_ERR_SIZE: return "a size argument is out of range";
        case MLA_ERR_WORKSPACE: return "workspace is smaller than mla_sparse_decode_workspace_size()";
        case MLA_ERR_CUDA: return "a CUDA launch or query failed";
        case MLA_ERR_DEVICE: return "the current device is not an sm_103 GPU";
        default: break;
    }
    if (code > 0) {
        static const char *names[8] = {"none",
                                       "bad end_pos",
                                       "position outside rotary table",
                                       "bad end_pos; position outside rotary table",
                                       "on-chip wait timed out",
                                       "bad end_pos; on-chip wait timed out",
                                       "position outside rotary table; on-chip wait timed out",
                                       "bad end_pos; position outside rotary table; on-chip wait timed out"};
        return names[code & 7];
    }
    return "unknown status code";
}
