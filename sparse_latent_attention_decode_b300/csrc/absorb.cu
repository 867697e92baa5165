// Query of the latent attention: key absorption on the tensor cores, with the
// RoPE of q_pe fused in.
//
// Source: DeepSeek-V3.2-Exp atlas, "Query content heads" page, excerpt
// mla-decode (first einsum: q_nope . W_UK per head), and "Rotated query part"
// page, excerpt apply-rope (pair rotation of q_pe).
//
// One CTA per (latent tile t, head h) computes, in the transposed
// ("swap-AB") form that puts 128 latent columns on the MMA rows,
//     q~_h^T [128t .. 128t+127, B] = W_UK[h][:, tile]^T [128, 128] . q_nope_h^T [128, B]
// with N = the batch (up to 128 sequences per pass): 512 CTAs of 128
// threads.  The W_UK tile (32 KB) arrives by TMA and is read MN-major; the
// batch tile arrives K-major through a 3-D tensor map over q_nope.  While the
// copies are in flight, the CTA rotates pairs 8t .. 8t+7 of q_pe for every
// sequence.  Results leave TMEM as bf16 rows of q_lat.
#include "common.cuh"
#include "kernels.cuh"
#include "tc05.cuh"

namespace mla {
namespace absorb {

using namespace tc;

constexpr int NMAX = 128;                      // sequences per pass, at most
constexpr int A_BOX = 128 * 128;               // one [128 d][64 c] box of W_UK, bytes
constexpr int B_BOX = NMAX * 128;              // one [128 b][64 d] box of q_nope, bytes, at most
constexpr int SMEM_BYTES = 2 * A_BOX + 2 * B_BOX + 1024;
// Shared memory for `nmax` sequences per pass: with B <= 64 four CTAs fit on
// an SM, so the 512 CTAs run as one wave.
__host__ __device__ constexpr int smem_bytes(int nmax) { return 2 * A_BOX + 2 * nmax * 128 + 1024; }
constexpr int PAIRS_PER_TILE = NPAIR / 4;      // rotary pairs handled by each latent tile
struct Bars {
    uint64_t a_full, b_full, mma_done, drain;
    uint32_t tmem_base;
};

// Interleaved rotation of pairs [8t, 8t+8) of q_pe[b, h] for every query row,
// four items per thread at a time so that the loads overlap.  Row b is token
// b % T of sequence b / T, at position end_pos[b / T] - T + b % T.
__device__ __forceinline__ void rope_part(const uint16_t *__restrict__ q_pe, const float2 *__restrict__ cis,
                                          int max_seq_len, const int32_t *__restrict__ end_pos, int B, int T,
                                          int h, int t, uint16_t *__restrict__ q_lat, int32_t *status, int tid) {
    constexpr int BATCH = 4;
    const int total = B * PAIRS_PER_TILE;
    for (int k0 = tid; k0 < total; k0 += 128 * BATCH) {
        int pos[BATCH];
#pragma unroll
        for (int u = 0; u < BATCH; ++u) {
            const int k = k0 + 128 * u;
            const int row = k / PAIRS_PER_TILE, seq = row / T;
            pos[u] = k < total ? end_pos[seq] - T + (row - seq * T) : -1;
        }
        uint32_t w[BATCH];
        float2 cs[BATCH];
#pragma unroll
        for (int u = 0; u < BATCH; ++u) {
            const int k = k0 + 128 * u;
            const int b = k / PAIRS_PER_TILE, i = PAIRS_PER_TILE * t + k % PAIRS_PER_TILE;
            const bool in = k < total && pos[u] >= 0 && pos[u] < max_seq_len;
            w[u] = in ? reinterpret_cast<const uint32_t *>(q_pe + ((size_t)b * H + h) * DR)[i] : 0u;
            cs[u] = in ? cis[(size_t)pos[u] * NPAIR + i] : make_float2(0.f, 0.f);
        }
#pragma unroll
        for (int u = 0; u < BATCH; ++u) {
            const int k = k0 + 128 * u;
            if (k >= total) continue;
            const int b = k / PAIRS_PER_TILE, i = PAIRS_PER_TILE * t + k % PAIRS_PER_TILE;
            const float x0 = bflo(w[u]), x1 = bfhi(w[u]);
            const uint32_t packed = uint32_t(f2bf(x0 * cs[u].x - x1 * cs[u].y)) |
                                    (uint32_t(f2bf(x0 * cs[u].y + x1 * cs[u].x)) << 16);
            reinterpret_cast<uint32_t *>(q_lat + ((size_t)b * H + h) * QL + C)[i] = packed;
            if ((pos[u] < 0 || pos[u] >= max_seq_len) && i == 0 && h == 0) report(status, MLA_DEV_BAD_POSITION);
        }
    }
}

__global__ void __launch_bounds__(128, 4)
    absorb_kernel(const __grid_constant__ CUtensorMap wmap, const __grid_constant__ CUtensorMap qmap,
                  const uint16_t *__restrict__ q_pe, const float2 *__restrict__ cis, int max_seq_len,
                  const int32_t *__restrict__ end_pos, int B, int T, int nmax, uint16_t *__restrict__ q_lat,
                  int32_t *status, uint64_t wait_ns) {
    extern __shared__ uint8_t smem_raw[];
    __shared__ Bars bars;
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *sA = smem, *sB = smem + 2 * A_BOX;
    const int t = blockIdx.x, h = blockIdx.y, tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    const int bbox = nmax * 128;   // bytes of one [nmax b][64 d] box of q_nope
    const int npass = (B + nmax - 1) / nmax;
    int b_issued = 0;   // batch tiles whose loads tid 0 has issued
    if (tid == 0) {
        mbar_init(&bars.a_full, 1);
        mbar_init(&bars.b_full, 1);
        mbar_init(&bars.mma_done, 1);
        mbar_init(&bars.drain, 1);
        fence_mbar_init();
        // the copies go out first, before the TMEM allocation and the CTA barrier:
        // W_UK[h] = rows h*256 .. h*256+127 of wkv_b, this tile = latent columns
        // 128t .. 128t+127; then the first batch tile of q_nope
        mbar_expect_tx(&bars.a_full, 2 * A_BOX);
        tma_load_2d(smem_u32(sA), &wmap, 128 * t, h * WROWS, &bars.a_full);
        tma_load_2d(smem_u32(sA + A_BOX), &wmap, 128 * t + 64, h * WROWS, &bars.a_full);
        mbar_expect_tx(&bars.b_full, 2 * bbox);
        tma_load_3d(smem_u32(sB), &qmap, 0, h, 0, &bars.b_full);
        tma_load_3d(smem_u32(sB + bbox), &qmap, 64, h, 0, &bars.b_full);
        b_issued = 1;
    }
    if (warp == 0) {
        tmem_alloc(&bars.tmem_base, NMAX);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    // the attention grid may be scheduled as soon as every CTA of this one has started
    if (tid == 0) grid_dep_launch();
    const uint32_t tmem = bars.tmem_base;
    const Deadline deadline = make_deadline(wait_ns);
    bool ok = true;

    for (int pass = 0; pass < npass && ok; ++pass) {
        const int n0 = pass * nmax;
        const int nb = min(nmax, B - n0);
        const int N = (nb + 15) & ~15;
        if (tid == 0 && pass > 0) {
            mbar_expect_tx(&bars.b_full, 2 * bbox);
            tma_load_3d(smem_u32(sB), &qmap, 0, h, n0, &bars.b_full);
            tma_load_3d(smem_u32(sB + bbox), &qmap, 64, h, n0, &bars.b_full);
            b_issued = pass + 1;
        }
        if (pass == 0) rope_part(q_pe, cis, max_seq_len, end_pos, B, T, h, t, q_lat, status, tid);
        if (tid == 0) {
            bool good = wait_until(&bars.b_full, pass & 1, deadline);
            if (pass == 0) good = good && wait_until(&bars.a_full, 0, deadline);
            if (good) {
                tc_fence_after();
                const uint32_t idesc = idesc_bf16(128, N, true, false);
#pragma unroll
                for (int kk = 0; kk < 8; ++kk) {
                    const uint64_t ad = smem_desc(smem_u32(sA) + kk * 2048, A_BOX, 1024, 2);
                    const uint64_t bd = smem_desc(smem_u32(sB + (kk >> 2) * bbox) + (kk & 3) * 32, 16, 1024, 2);
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
        // epilogue: lane = latent column within the tile, column = query row.  The
        // rows are staged in shared memory over the batch tile (its MMAs have
        // completed; row pitch 256 B, each warp writing 64 contiguous bytes of a
        // row at a time) and leave as whole 256-byte row segments of q_lat.
        {
            const uint32_t trow = tmem + (uint32_t(32 * warp) << 16);
            const uint32_t stg = smem_u32(sB) + (32 * warp + lane) * 2;
            for (int j0 = 0; j0 < N; j0 += 16) {
                uint32_t v[16];
                tmem_ld16(trow + j0, v);
                tmem_ld_wait();
#pragma unroll
                for (int i = 0; i < 16; ++i)
                    asm volatile("st.shared.b16 [%0], %1;" ::"r"(stg + (j0 + i) * 256), "h"(f2bf(__uint_as_float(v[i])))
                                 : "memory");
            }
        }
        __syncthreads();
        for (int idx = tid; idx < nb * 16; idx += 128) {
            const int row = idx >> 4, ch = idx & 15;
            uint32_t a0, a1, a2, a3;
            asm volatile("ld.shared.v4.b32 {%0,%1,%2,%3}, [%4];"
                         : "=r"(a0), "=r"(a1), "=r"(a2), "=r"(a3)
                         : "r"(smem_u32(sB) + row * 256 + ch * 16));
            *reinterpret_cast<uint4 *>(q_lat + ((size_t)(n0 + row) * H + h) * QL + 128 * t + ch * 8) =
                make_uint4(a0, a1, a2, a3);
        }
        // the next pass's batch tile overwrites the staging by TMA (async proxy)
        fence_proxy_async_smem();
        tc_fence_before();
        __syncthreads();   // TMEM and the batch tile are reused by the next pass
    }
    if (!ok && tid == 0) report(status, MLA_DEV_TIMEOUT);
    if (tid == 0) {
        // drain: the weight tile and the last batch tile have landed and every
        // issued MMA has completed before the CTA releases TMEM and exits
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

}  // namespace absorb
}  // namespace mla

using namespace mla;

extern "C" int mla_absorb_q_tokens(const mla_bf16 *q_nope, const mla_bf16 *q_pe, const float *cis,
                                   int max_seq_len, const int32_t *end_pos, const mla_bf16 *wkv_b, int n_seq, int T,
                                   mla_bf16 *q_lat, int32_t *dev_status, mla_stream_t stream) {
    if (!q_nope || !q_pe || !cis || !end_pos || !wkv_b || !q_lat) return MLA_ERR_NULL;
    if (!aligned16(q_nope) || !aligned16(q_pe) || !aligned16(cis) || !aligned16(wkv_b) || !aligned16(q_lat))
        return MLA_ERR_ALIGN;
    if (n_seq < 1 || T < 1 || (long long)n_seq * T > 4096 || max_seq_len < 1) return MLA_ERR_SIZE;
    const int B = n_seq * T;   // query rows
    const int nmax = B >= absorb::NMAX ? absorb::NMAX : (B + 15) / 16 * 16;
    CUtensorMap wmap, qmap;
    {
        const uint64_t dims[2] = {(uint64_t)C, (uint64_t)H * WROWS};
        const uint64_t strides[1] = {(uint64_t)C * 2};
        const uint32_t box[2] = {64, 128};
        if (!make_tmap_bf16(&wmap, wkv_b, 2, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B)) return MLA_ERR_CUDA;
    }
    {
        const uint64_t dims[3] = {(uint64_t)DN, (uint64_t)H, (uint64_t)B};
        const uint64_t strides[2] = {(uint64_t)DN * 2, (uint64_t)H * DN * 2};
        const uint32_t box[3] = {64, 1, (uint32_t)nmax};
        if (!make_tmap_bf16(&qmap, q_nope, 3, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B)) return MLA_ERR_CUDA;
    }
    cudaStream_t s = (cudaStream_t)stream;
    static std::atomic<bool> smem_set[64];
    if (!smem_attr_once(smem_set, absorb::absorb_kernel, absorb::SMEM_BYTES)) return MLA_ERR_CUDA;
    absorb::absorb_kernel<<<dim3(4, H), 128, absorb::smem_bytes(nmax), s>>>(
        wmap, qmap, q_pe, reinterpret_cast<const float2 *>(cis), max_seq_len, end_pos, B, T, nmax, q_lat, dev_status,
        wait_limit_ns());
    count_launches(1);
    return cudaGetLastError() == cudaSuccess ? MLA_OK : MLA_ERR_CUDA;
}

extern "C" int mla_absorb_q(const mla_bf16 *q_nope, const mla_bf16 *q_pe, const float *cis, int max_seq_len,
                            const int32_t *end_pos, const mla_bf16 *wkv_b, int B, mla_bf16 *q_lat,
                            int32_t *dev_status, mla_stream_t stream) {
    return mla_absorb_q_tokens(q_nope, q_pe, cis, max_seq_len, end_pos, wkv_b, B, 1, q_lat, dev_status, stream);
}
