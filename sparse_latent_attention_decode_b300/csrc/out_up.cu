// Value up-projection on the tensor cores: out[b,h,d] = sum_c o[b,h,c] * W_UV[h][d][c].
//
// Source: DeepSeek-V3.2-Exp atlas, "Attention weights" page, excerpt
// mla-decode (last einsum, wkv_b[:, -v_head_dim:]).
//
// One CTA per head h computes out_h^T [128 d, B] = W_UV[h] [128, 512] . o_h^T
// [512, B] ("swap-AB": the head's 128 output features fill the MMA rows, the
// batch is N), 64 sequences per pass.  W_UV[h] (128 KB) is loaded once by TMA
// (K-major).  The latent outputs o arrive either as bf16 (written by the
// attention kernel; loaded by TMA through a 3-D tensor map) or as fp32 (the
// standalone entry point; rounded to bf16 while they are written into the
// 128-byte-swizzled operand tile).  The one or two query rows of a split
// selection are merged from the split partials and stay fp32: their product
// with W_UV runs on the CUDA cores (a 16-column MMA pass is bound by the issue
// of its 32 instructions).
//
// The kernel is launched as a programmatic dependent of the attention grid.
// It loads W_UV before griddepcontrol.wait: the attention grid itself waits
// for every grid before it before it lets this one start, and it does not
// write W_UV, so W_UV is final by then.  o is read only after the wait.
#include "common.cuh"
#include "kernels.cuh"
#include "tc05.cuh"

namespace mla {
namespace outup {

using namespace tc;

constexpr int NMAX = 64;                       // sequences per pass
constexpr int A_BOX = 128 * 128;               // [128 d][64 c] box of W_UV, bytes
constexpr int B_ATOM = NMAX * 128;             // [64 b][64 c] atom column of the o tile, bytes
constexpr int SMEM_BYTES = 8 * A_BOX + 8 * B_ATOM + 1024;
constexpr int MERGE_ROWS = 2, MERGE_SPLITS = 128;   // split partials merged here: rows and splits per row, at most
struct Bars {
    uint64_t a_full, b_full, mma_done, drain;
    uint32_t tmem_base;
};

// fp32 o rows of one pass -> bf16 operand tile: 16-byte chunk (row, c/8), 64
// chunks per row; loads are issued eight chunks at a time so that their
// latencies overlap.
__device__ __forceinline__ void stage_f32(const float *__restrict__ o_lat, int h, int n0, int nb, int N,
                                          uint8_t *sB, int tid) {
    constexpr int BATCH = 8;
    const int total = N * 64;
    for (int u0 = tid; u0 < total; u0 += 128 * BATCH) {
        float4 x[BATCH][2];
#pragma unroll
        for (int k = 0; k < BATCH; ++k) {
            const int u = u0 + 128 * k, row = u >> 6, ch = u & 63;
            if (u < total && row < nb) {
                const float4 *src = reinterpret_cast<const float4 *>(o_lat + ((size_t)(n0 + row) * H + h) * C + ch * 8);
                x[k][0] = src[0];
                x[k][1] = src[1];
            } else {
                x[k][0] = x[k][1] = make_float4(0.f, 0.f, 0.f, 0.f);
            }
        }
#pragma unroll
        for (int k = 0; k < BATCH; ++k) {
            const int u = u0 + 128 * k, row = u >> 6, ch = u & 63;
            if (u < total)
                *reinterpret_cast<uint4 *>(sB + (ch >> 3) * B_ATOM + sw128(row, ch & 7)) =
                    make_uint4(pack_bf16(x[k][0].x, x[k][0].y), pack_bf16(x[k][0].z, x[k][0].w),
                               pack_bf16(x[k][1].x, x[k][1].y), pack_bf16(x[k][1].z, x[k][1].w));
        }
    }
}

// Split partials -> fp32 rows o_s [nb][512], for the one or two query rows of
// a split selection: each row's latent output o is merged from its n_split
// partials (normalised o of every split as bf16, and the log2 of each split's
// softmax mass, one per latent half and head), o = sum_s 2^(lse_s - M) o_s /
// sum_s 2^(lse_s - M) with M the largest lse_s, as the split-combine kernel
// merges them (in fp32).  One warp per (row, half) turns the masses into
// normalised weights in shared memory; then each thread sums four latent
// columns of a row over the splits, with the loads of several splits in
// flight at once.
__device__ __forceinline__ void stage_partials(const uint16_t *__restrict__ part_o, const float *__restrict__ part_lse,
                                               int n_split, int h, int n0, int nb, float *o_s, int tid,
                                               float (*wts)[2][MERGE_SPLITS]) {
    const int warp = tid >> 5, lane = tid & 31;
    {
        const int row = warp >> 1, half = warp & 1;   // four warps: rows 0..1, halves 0..1
        if (row < nb) {
            // each lane holds the masses of splits lane, lane+32, ... (one load each)
            constexpr int PER_LANE = MERGE_SPLITS / 32;
            const size_t u0 = (size_t)(n0 + row) * n_split;
            float lse[PER_LANE];
            float M = -INFINITY;
#pragma unroll
            for (int k = 0; k < PER_LANE; ++k) {
                const int sp = lane + 32 * k;
                lse[k] = sp < n_split ? part_lse[((u0 + sp) * 2 + half) * H + h] : -INFINITY;
                M = fmaxf(M, lse[k]);
            }
#pragma unroll
            for (int off = 16; off; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
            float L = 0.f;
#pragma unroll
            for (int k = 0; k < PER_LANE; ++k) {
                lse[k] = (M == -INFINITY || lse[k] == -INFINITY) ? 0.f : exp2f(lse[k] - M);   // now the weight
                L += lse[k];
            }
#pragma unroll
            for (int off = 16; off; off >>= 1) L += __shfl_xor_sync(0xffffffffu, L, off);
            const float inv = L > 0.f ? 1.f / L : 0.f;
#pragma unroll
            for (int k = 0; k < PER_LANE; ++k)
                if (lane + 32 * k < n_split) wts[row][half][lane + 32 * k] = lse[k] * inv;
        }
    }
    __syncthreads();
    // piece q (4 latent columns) of row `row`: 128 per row, 8 bytes of partial, 16 of the merged row
    for (int u = tid; u < nb * 128; u += 128) {
        const int row = u >> 7, q = u & 127, half = q >= 64 ? 1 : 0;
        float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
        if (row < nb) {
            const float *w = wts[row][half];
            const uint2 *src = reinterpret_cast<const uint2 *>(part_o + ((size_t)(n0 + row) * n_split * H + h) * C) + q;
            constexpr size_t STEP = (size_t)H * C / 4;   // 4-element pieces between two splits of the row
#pragma unroll 16
            for (int sp = 0; sp < n_split; ++sp) {
                // an empty split has weight 0 and a zero o (its unit writes zeros), so
                // every split is loaded unconditionally and the loads go out together
                const float ws = w[sp];
                const uint2 v = src[sp * STEP];
                a.x = fmaf(ws, bflo(v.x), a.x), a.y = fmaf(ws, bfhi(v.x), a.y);
                a.z = fmaf(ws, bflo(v.y), a.z), a.w = fmaf(ws, bfhi(v.y), a.w);
            }
        }
        *reinterpret_cast<float4 *>(o_s + row * C + 4 * q) = a;
    }
}

__global__ void __launch_bounds__(128, 1) out_up_kernel(const __grid_constant__ CUtensorMap wmap,
                                                        const __grid_constant__ CUtensorMap omap,
                                                        const float *__restrict__ o_f32, bool o_is_b16, int B,
                                                        const uint16_t *__restrict__ part_o,
                                                        const float *__restrict__ part_lse, int n_split,
                                                        float *__restrict__ out, uint16_t *__restrict__ out_b16,
                                                        int32_t *status, uint64_t wait_ns) {
    extern __shared__ uint8_t smem_raw[];
    __shared__ Bars bars;
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *sA = smem, *sB = smem + 8 * A_BOX;
    const int h = blockIdx.x, tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    if (tid == 0) {
        mbar_init(&bars.a_full, 1);
        mbar_init(&bars.b_full, 1);
        mbar_init(&bars.mma_done, 1);
        mbar_init(&bars.drain, 1);
        fence_mbar_init();
    }
    if (warp == 0) {
        tmem_alloc(&bars.tmem_base, NMAX);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = bars.tmem_base;
    const Deadline deadline = make_deadline(wait_ns);
    int b_issued = 0;   // o tiles whose loads tid 0 has issued

    if (tid == 0) {   // W_UV[h] = rows h*256+128 .. h*256+255 of wkv_b, 8 boxes of 64 latent columns
        mbar_expect_tx(&bars.a_full, 8 * A_BOX);
        for (int a = 0; a < 8; ++a)
            tma_load_2d(smem_u32(sA + a * A_BOX), &wmap, 64 * a, h * WROWS + DN, &bars.a_full);
    }
    grid_dep_wait();   // o is written by the preceding grid

    bool ok = true;
    const int npass = (B + NMAX - 1) / NMAX;
    for (int pass = 0; pass < npass && ok; ++pass) {
        const int n0 = pass * NMAX;
        const int nb = min(NMAX, B - n0);
        const int N = (nb + 15) & ~15;
        if (o_is_b16) {
            if (tid == 0) {   // 8 boxes [64 b][64 c] of o_h; rows beyond B are zero-filled
                mbar_expect_tx(&bars.b_full, 8 * B_ATOM);
                for (int a = 0; a < 8; ++a) tma_load_3d(smem_u32(sB + a * B_ATOM), &omap, 64 * a, h, n0, &bars.b_full);
                b_issued = pass + 1;
            }
        } else if (part_o) {
            // one or two query rows from split partials: the merged rows stay fp32 and
            // each thread takes one output feature d, a dot product of its W_UV row (in
            // shared memory, 128B-swizzled boxes of 64 latent columns) with each row on
            // the CUDA cores -- at N = 16 the 32 tensor-core MMAs are bound by their issue
            // (about 1.5 us), the dot products take a fraction of that
            __shared__ float wts[MERGE_ROWS][2][MERGE_SPLITS];
            __shared__ __align__(16) float o_s[MERGE_ROWS * C];
            stage_partials(part_o, part_lse, n_split, h, n0, nb, o_s, tid, wts);
            ok = __syncthreads_and(wait_until(&bars.a_full, 0, deadline));
            if (!ok) break;
            const int d = tid;
            float acc[MERGE_ROWS];
#pragma unroll
            for (int rw = 0; rw < MERGE_ROWS; ++rw) acc[rw] = 0.f;
#pragma unroll 1
            for (int a = 0; a < 8; ++a) {   // box a: latent columns 64a .. 64a+63
                const uint8_t *wr = sA + a * A_BOX + d * 128;
#pragma unroll
                for (int j = 0; j < 8; ++j) {   // chunk j: columns 64a+8j .. 64a+8j+7
                    const uint4 wv = *reinterpret_cast<const uint4 *>(wr + ((j ^ (d & 7)) << 4));
                    const float w[8] = {bflo(wv.x), bfhi(wv.x), bflo(wv.y), bfhi(wv.y),
                                        bflo(wv.z), bfhi(wv.z), bflo(wv.w), bfhi(wv.w)};
#pragma unroll
                    for (int rw = 0; rw < MERGE_ROWS; ++rw) {
                        if (rw >= nb) break;
                        const float4 o0 = *reinterpret_cast<const float4 *>(o_s + rw * C + 64 * a + 8 * j);
                        const float4 o1 = *reinterpret_cast<const float4 *>(o_s + rw * C + 64 * a + 8 * j + 4);
                        float s = acc[rw];
                        s = fmaf(w[0], o0.x, s), s = fmaf(w[1], o0.y, s), s = fmaf(w[2], o0.z, s);
                        s = fmaf(w[3], o0.w, s), s = fmaf(w[4], o1.x, s), s = fmaf(w[5], o1.y, s);
                        s = fmaf(w[6], o1.z, s), s = fmaf(w[7], o1.w, s);
                        acc[rw] = s;
                    }
                }
            }
#pragma unroll
            for (int rw = 0; rw < MERGE_ROWS; ++rw) {
                if (rw >= nb) break;
                const size_t at = ((size_t)(n0 + rw) * H + h) * DV + d;
                if (out_b16)
                    out_b16[at] = f2bf(acc[rw]);
                else
                    out[at] = acc[rw];
            }
            continue;   // no tensor-core pass for these rows
        } else {
            stage_f32(o_f32, h, n0, nb, N, sB, tid);
            fence_proxy_async_smem();
        }
        __syncthreads();
        if (tid == 0) {
            bool good = (pass > 0 || wait_until(&bars.a_full, 0, deadline)) &&
                        (!o_is_b16 || wait_until(&bars.b_full, pass & 1, deadline));
            if (good) {
                tc_fence_after();
                const uint32_t idesc = idesc_bf16(128, N, false, false);
#pragma unroll 4
                for (int kk = 0; kk < 32; ++kk) {
                    const uint64_t ad = smem_desc(smem_u32(sA + (kk >> 2) * A_BOX) + (kk & 3) * 32, 16, 1024, 2);
                    const uint64_t bd = smem_desc(smem_u32(sB + (kk >> 2) * B_ATOM) + (kk & 3) * 32, 16, 1024, 2);
                    mma_ss(tmem, ad, bd, idesc, kk > 0);
                }
                mma_commit(&bars.mma_done);
            } else {
                report(status, MLA_DEV_TIMEOUT);
            }
        }
        ok = __syncthreads_and(wait_until(&bars.mma_done, pass & 1, deadline));
        if (!ok) break;
        tc_fence_after();
        const uint32_t trow = tmem + (uint32_t(32 * warp) << 16);
        const int d = 32 * warp + lane;
        for (int j0 = 0; j0 < N; j0 += 16) {
            uint32_t v[16];
            tmem_ld16(trow + j0, v);
            tmem_ld_wait();
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                const int b = n0 + j0 + i;
                if (b >= B) continue;
                const size_t at = ((size_t)b * H + h) * DV + d;
                if (out_b16)
                    out_b16[at] = f2bf(__uint_as_float(v[i]));
                else
                    out[at] = __uint_as_float(v[i]);
            }
        }
        tc_fence_before();
        __syncthreads();   // TMEM and the operand tile are reused by the next pass
    }
    if (!ok && tid == 0) report(status, MLA_DEV_TIMEOUT);
    if (tid == 0) {
        // drain: W_UV and the last o tile have landed and every issued MMA has
        // completed before the CTA releases TMEM and exits
        const uint64_t drain = globaltimer_ns() + DRAIN_NS;
        bool landed = wait_until(&bars.a_full, 0, drain);
        if (b_issued > 0) landed = wait_until(&bars.b_full, (b_issued - 1) & 1, drain) && landed;
        mma_commit(&bars.drain);
        landed = wait_until(&bars.drain, 0, drain) && landed;
        if (!landed) report(status, MLA_DEV_TIMEOUT);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, NMAX);
    }
}

}  // namespace outup

int launch_out_up(const float *o_f32, const uint16_t *o_b16, const uint16_t *wkv_b, int B, float *out,
                  uint16_t *out_b16, int32_t *status, cudaStream_t s, bool pdl, const uint16_t *part_o,
                  const float *part_lse, int n_split) {
    CUtensorMap wmap, omap;
    {
        const uint64_t dims[2] = {(uint64_t)C, (uint64_t)H * WROWS};
        const uint64_t strides[1] = {(uint64_t)C * 2};
        const uint32_t box[2] = {64, 128};
        if (!make_tmap_bf16(&wmap, wkv_b, 2, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B)) return MLA_ERR_CUDA;
    }
    if (o_b16) {
        const uint64_t dims[3] = {(uint64_t)C, (uint64_t)H, (uint64_t)B};
        const uint64_t strides[2] = {(uint64_t)C * 2, (uint64_t)H * C * 2};
        const uint32_t box[3] = {64, 1, outup::NMAX};
        if (!make_tmap_bf16(&omap, o_b16, 3, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B)) return MLA_ERR_CUDA;
    } else {
        omap = wmap;   // unused
    }
    // split partials are merged here only for the one or two rows of a split selection
    if (part_o && (B > outup::MERGE_ROWS || n_split < 1 || n_split > outup::MERGE_SPLITS)) return MLA_ERR_SIZE;
    static std::atomic<bool> smem_set[64];
    if (!smem_attr_once(smem_set, outup::out_up_kernel, outup::SMEM_BYTES)) return MLA_ERR_CUDA;
    const cudaError_t err = launch_k(pdl, outup::out_up_kernel, dim3(H), dim3(128), outup::SMEM_BYTES, s, wmap,
                                     omap, o_f32, o_b16 != nullptr, B, part_o, part_lse, n_split, out, out_b16, status,
                                     wait_limit_ns());
    count_launches(1);
    return err == cudaSuccess ? MLA_OK : MLA_ERR_CUDA;
}

}  // namespace mla

using namespace mla;

extern "C" int mla_out_up(const float *o_lat, const mla_bf16 *wkv_b, int B, float *out, mla_stream_t stream) {
    if (!o_lat || !wkv_b || !out) return MLA_ERR_NULL;
    if (!aligned16(o_lat) || !aligned16(wkv_b) || !aligned16(out)) return MLA_ERR_ALIGN;
    if (B < 1 || B > 4096) return MLA_ERR_SIZE;
    return launch_out_up(o_lat, nullptr, wkv_b, B, out, nullptr, nullptr, (cudaStream_t)stream, false);
}
