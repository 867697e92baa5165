// Sparse latent attention on the 5th-generation tensor cores (tcgen05 + TMEM),
// fed by 16-byte cp.async row gathers.
//
// Source: DeepSeek-V3.2-Exp atlas, "Attention weights" page, excerpt
// mla-decode: scores = (q~ . kv + q_pe . pe) * scale over the cached rows,
// -inf outside the selected set, softmax over keys, probabilities . kv.
//
// Work unit: one sequence b (or one split of its selection), processed by a
// cluster of two CTAs that split the 576-wide contraction and the 512-wide
// latent output between them:
//   CTA r gathers, for every selected key, latent columns [256r, 256r+256)
//   and rotary columns [32r, 32r+32) -- each byte of a selected row is read
//   from HBM exactly once by the pair.
//   QK  : S_r[128 heads, 64 keys] = Q_r . K_r^T  (A = Q_r resident in TMEM,
//         B = the gathered tile, K-major), 18 MMAs of K=16.
//   The two partial score tiles are exchanged through distributed shared
//   memory (fp16, scaled to log2 units) and summed: both CTAs then hold the
//   full scores and run the same online softmax (one thread per head).
//   PV  : O_r[128 heads, 256 latent] += P[128, 64] . V_r[64, 256]  (A = P
//         in TMEM as bf16, B = the same gathered tile read MN-major).
// TMEM per CTA: O_r 256 columns, Q_r 144, S 64, P 32 (512 allocated).
// The softmax keeps a running maximum per head that is raised only when a
// block's maximum exceeds it by more than 8 (log2 units); O and the running
// sum are rescaled then, which keeps every exponent <= 2^8 and is exact up to
// rounding because numerator and denominator share the same maximum.
#include "common.cuh"
#include "kernels.cuh"
#include "tc05.cuh"

#include <math.h>

namespace mla {
namespace attn {

using namespace tc;

constexpr int NK = 64;                       // keys per block
constexpr int NS = 5;                        // gather pipeline stages
constexpr int STAGE_KV = 4 * NK * 128;       // 4 atom columns of 64 latent x 64 keys (128B swizzle)
constexpr int STAGE_PE = NK * 64;            // 32 rotary columns x 64 keys (64B swizzle)
constexpr int STAGE = STAGE_KV + STAGE_PE;   // 36864
constexpr int RECV = H * NK * 2;             // fp16 partial scores of the peer, 128 x 64
constexpr int SMEM_BYTES = NS * STAGE + 2 * RECV + 1024;
constexpr uint32_t O_COL = 0, Q_COL = 256, S_COL = 400, P_COL = 464, TMEM_COLS = 512;
// warps 0..7 gather (cp.async), 8..11 softmax, 12 MMA, 13..15 idle: four
// warpgroups, so that registers can move from the gather warps to the softmax
constexpr int THREADS = 512;
constexpr int GATHER_THREADS = 256;
constexpr int CHUNKS = NK * 36;              // 16-byte chunks per stage: 32 latent + 4 rotary per key
constexpr int CHUNKS_PER_THREAD = CHUNKS / GATHER_THREADS;   // 9
constexpr int MMA_WARP = 12;
// A gather thread publishes block j once it has issued block j+LAG and the
// copies of block j have landed.  The MMA issues QK two blocks ahead of PV, so
// block j+2 must be published without waiting for a stage that PV(j) frees:
// (j + 2 + LAG) - NS < j, i.e. LAG <= NS - 3.
constexpr int LAG = 2;
static_assert(LAG <= NS - 3, "gather publication lag would deadlock against the QK lookahead");
constexpr float RESCALE_T = 8.f;             // lazy-max threshold (log2 units)
constexpr uint64_t TIMEOUT_NS = 2000000000ull;

struct Params {
    const uint16_t *q_lat;
    const uint16_t *kv;
    const uint16_t *pe;
    const int32_t *topk;
    const int32_t *end_pos;
    int S_cap, K, B;
    float scale_log2;   // softmax_scale * log2(e)
    int n_split, split_len;
    float *o_out;       // n_split == 1: normalised o, fp32 [B][128][512]
    float *part_o;      // n_split > 1: per-split normalised o, fp32 [B*n_split][128][512]
    float *part_lse;    // n_split > 1: log2 of the split's softmax mass, [B*n_split][2][128]
    int32_t *status;
};

struct Bars {
    uint64_t full[NS], empty[NS];
    uint64_t s_full, s_free, p_full, pv_done, q_ready;
    uint64_t recv_full[2], send_credit[2];
    uint32_t tmem_base;
};

__device__ __forceinline__ void fail(const Params &p) { report(p.status, MLA_DEV_TIMEOUT); }

// warp-uniform bounded waits: every lane of the warp takes the same branch afterwards
__device__ __forceinline__ bool warp_wait(uint64_t *bar, uint32_t parity, uint64_t deadline) {
    return __all_sync(0xffffffffu, wait_until(bar, parity, deadline));
}
__device__ __forceinline__ bool warp_wait_cluster(uint64_t *bar, uint32_t parity, uint64_t deadline) {
    return __all_sync(0xffffffffu, wait_until_cluster(bar, parity, deadline));
}

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(THREADS, 1) attn_kernel(Params p) {
    extern __shared__ uint8_t smem_raw[];
    __shared__ Bars bars;
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *stages = smem;
    uint8_t *recv = smem + NS * STAGE;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const uint32_t r = cluster_rank(), peer = r ^ 1u;
    const int unit = blockIdx.x >> 1;
    const int b = unit / p.n_split, split = unit % p.n_split;
    const int e = p.end_pos[b];
    const bool seq_ok = e >= 1 && e <= p.S_cap;
    const int t0 = split * p.split_len;
    const int t1 = min(p.K, t0 + p.split_len);
    const int nblk = (seq_ok && t1 > t0) ? (t1 - t0 + NK - 1) / NK : 0;
    if (!seq_ok && tid == 0 && r == 0 && split == 0) report(p.status, MLA_DEV_BAD_END_POS);

    if (tid == 0) {
        for (int s = 0; s < NS; ++s) mbar_init(&bars.full[s], GATHER_THREADS), mbar_init(&bars.empty[s], 1);
        mbar_init(&bars.s_full, 1);
        mbar_init(&bars.s_free, 128);
        mbar_init(&bars.p_full, 128);
        mbar_init(&bars.pv_done, 1);
        mbar_init(&bars.q_ready, 128);
        for (int k = 0; k < 2; ++k) mbar_init(&bars.recv_full[k], 128), mbar_init(&bars.send_credit[k], 128);
        fence_mbar_init();
    }
    if (warp == MMA_WARP) {
        tmem_alloc(&bars.tmem_base, TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    cluster_sync();   // barriers of both CTAs initialised, TMEM address published
    tc_fence_after();
    const uint32_t tmem = bars.tmem_base;
    const uint64_t deadline = globaltimer_ns() + TIMEOUT_NS;

    if (warp < 8) {
        // ------------------------------------------------------------ gather producers
        // 256 threads copy a stage's 2304 16-byte chunks with cp.async, 9 each.
        // Chunk e = tid + 256 q belongs to key e / 36; chunks 0..31 of a key are
        // its latent half (4 atom columns x 8, 128-byte swizzle), 32..35 its
        // rotary half (64-byte swizzle).  Invalid keys are zero-filled.
        regs_dec<96>();
        uint32_t dst_off[CHUNKS_PER_THREAD];
        int src_off[CHUNKS_PER_THREAD], key[CHUNKS_PER_THREAD];
        bool is_pe[CHUNKS_PER_THREAD];
#pragma unroll
        for (int q = 0; q < CHUNKS_PER_THREAD; ++q) {
            const int ch = tid + GATHER_THREADS * q;
            key[q] = ch / 36;
            const int c = ch % 36;
            is_pe[q] = c >= 32;
            if (c < 32) {
                const int a = c >> 3, cc = c & 7;
                dst_off[q] = a * (NK * 128) + sw128(key[q], cc);
                src_off[q] = 256 * r + 64 * a + 8 * cc;
            } else {
                const int cc = c - 32;
                dst_off[q] = STAGE_KV + sw64(key[q], cc);
                src_off[q] = 32 * r + 8 * cc;
            }
        }
        const uint16_t *kvb = p.kv + (size_t)b * p.S_cap * C;
        const uint16_t *peb = p.pe + (size_t)b * p.S_cap * DR;
        const int32_t *sel = p.topk + (size_t)b * p.K;
        int cur[CHUNKS_PER_THREAD], nxt[CHUNKS_PER_THREAD];
        auto load_idx = [&](int j, int(&dst)[CHUNKS_PER_THREAD]) {
#pragma unroll
            for (int q = 0; q < CHUNKS_PER_THREAD; ++q) {
                const int slot = t0 + j * NK + key[q];
                const int id = slot < t1 ? sel[slot] : -1;
                dst[q] = (id >= 0 && id < e) ? id : -1;
            }
        };
        if (nblk > 0) load_idx(0, nxt);
        int j = 0;
        for (; j < nblk; ++j) {
#pragma unroll
            for (int q = 0; q < CHUNKS_PER_THREAD; ++q) cur[q] = nxt[q];
            if (j + 1 < nblk) load_idx(j + 1, nxt);   // prefetch: used next iteration
            const int s = j % NS;
            if (j >= NS && !warp_wait(&bars.empty[s], ((j / NS) - 1) & 1, deadline)) {
                fail(p);
                break;
            }
            const uint32_t base = smem_u32(stages + s * STAGE);
#pragma unroll
            for (int q = 0; q < CHUNKS_PER_THREAD; ++q) {
                const int row = cur[q] < 0 ? 0 : cur[q];
                const uint16_t *src = is_pe[q] ? peb + (size_t)row * DR + src_off[q] : kvb + (size_t)row * C + src_off[q];
                cp_async16(base + dst_off[q], src, cur[q] < 0 ? 0u : 16u);
            }
            cp_async_commit();
            if (j >= LAG) {   // the copies of block j-LAG have landed: publish them
                cp_async_wait<LAG>();
                fence_proxy_async_smem();
                mbar_arrive(&bars.full[(j - LAG) % NS]);
            }
        }
        cp_async_wait<0>();
        fence_proxy_async_smem();
        for (int jj = max(0, j - LAG); jj < j; ++jj) mbar_arrive(&bars.full[jj % NS]);
    } else if (warp >= 12) {
        // ------------------------------------------------------------ MMA issuer (warp 12, one thread)
        regs_dec<64>();
        if (warp == MMA_WARP && lane == 0 && nblk > 0) {
            bool ok = wait_until(&bars.q_ready, 0, deadline);
            tc_fence_after();
            constexpr uint32_t idesc_qk = idesc_bf16(128, NK, false, false);
            constexpr uint32_t idesc_pv = idesc_bf16(128, 256, false, true);
            auto issue_qk = [&](int j) -> bool {
                const int s = j % NS;
                if (!wait_until(&bars.full[s], (j / NS) & 1, deadline)) return false;
                if (j > 0 && !wait_until(&bars.s_free, (j - 1) & 1, deadline)) return false;
                tc_fence_after();
                const uint32_t base = smem_u32(stages + s * STAGE);
#pragma unroll
                for (int kk = 0; kk < 16; ++kk)
                    mma_ts(tmem + S_COL, tmem + Q_COL + kk * 8,
                           smem_desc(base + (kk >> 2) * (NK * 128) + (kk & 3) * 32, 16, 1024, 2), idesc_qk, kk > 0);
#pragma unroll
                for (int kk = 0; kk < 2; ++kk)
                    mma_ts(tmem + S_COL, tmem + Q_COL + 128 + kk * 8, smem_desc(base + STAGE_KV + kk * 32, 16, 512, 4),
                           idesc_qk, 1);
                mma_commit(&bars.s_full);
                return true;
            };
            auto issue_pv = [&](int j) -> bool {
                const int s = j % NS;
                if (!wait_until(&bars.p_full, j & 1, deadline)) return false;
                tc_fence_after();
                const uint32_t base = smem_u32(stages + s * STAGE);
#pragma unroll
                for (int kk = 0; kk < NK / 16; ++kk)
                    mma_ts(tmem + O_COL, tmem + P_COL + kk * 8, smem_desc(base + kk * 2048, NK * 128, 1024, 2),
                           idesc_pv, (j > 0 || kk > 0) ? 1u : 0u);
                mma_commit(&bars.pv_done);
                mma_commit(&bars.empty[s]);
                return true;
            };
            // QK runs two blocks ahead of PV: the softmax of block j overlaps QK(j+1)
            ok = ok && issue_qk(0);
            if (nblk > 1) ok = ok && issue_qk(1);
            for (int j = 0; ok && j < nblk; ++j) {
                if (j + 2 < nblk) ok = issue_qk(j + 2);
                ok = ok && issue_pv(j);
            }
            if (!ok) fail(p);
        }
    } else {
        // ------------------------------------------------------------ softmax warps (one thread per head)
        regs_inc<232>();
        const int quad = warp & 3;
        const int h = 32 * quad + lane;
        const uint32_t trow = tmem + (uint32_t(32 * quad) << 16);
        bool ok = true;
        float m = -INFINITY, l = 0.f;
        if (nblk > 0) {
            // Q_r -> TMEM: latent [256r, 256r+256) as 128 bf16 pairs, rotary [32r, 32r+32) as 16 pairs
            const uint4 *qrow = reinterpret_cast<const uint4 *>(p.q_lat + ((size_t)b * H + h) * QL);
#pragma unroll
            for (int c0 = 0; c0 < 9; ++c0) {
                uint32_t v[16];
                const int src16 = c0 < 8 ? (256 * r) / 8 + c0 * 4 : (512 + 32 * r) / 8;  // in 16-byte units
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const uint4 w = qrow[src16 + q];
                    v[4 * q] = w.x, v[4 * q + 1] = w.y, v[4 * q + 2] = w.z, v[4 * q + 3] = w.w;
                }
                tmem_st16(trow + Q_COL + 16 * c0, v);
            }
            tmem_st_wait();
            tc_fence_before();
            mbar_arrive(&bars.q_ready);
        }
        const uint32_t recv_local = smem_u32(recv);
        const uint32_t recv_peer = map_peer(recv_local, peer);
        const int32_t *sel = p.topk + (size_t)b * p.K;
        // Iteration j loads block j's partial scores and sends them to the peer,
        // then finishes block j-1, whose peer half arrived during the previous
        // iteration: the exchange latency hides behind a block of work.
        float xp[NK];
        uint32_t vpe = 0, vpo = 0;
        for (int j = 0; j <= nblk && ok; ++j) {
            float xc[NK];
            uint32_t vce = 0, vco = 0;
            if (j < nblk) {
                // validity of the block's 64 keys (key k: bit k/2 of vce for even k, of vco for odd k)
                const int slot = t0 + j * NK + 2 * lane;
                const int i0 = slot < t1 ? sel[slot] : -1;
                const int i1 = slot + 1 < t1 ? sel[slot + 1] : -1;
                vce = __ballot_sync(0xffffffffu, i0 >= 0 && i0 < e);
                vco = __ballot_sync(0xffffffffu, i1 >= 0 && i1 < e);

                if (!warp_wait(&bars.s_full, j & 1, deadline)) { ok = false; break; }
                tc_fence_after();
                {
                    uint32_t v[16];
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        tmem_ld16(trow + S_COL + 16 * c, v);
                        tmem_ld_wait();
#pragma unroll
                        for (int i = 0; i < 16; ++i) xc[16 * c + i] = __uint_as_float(v[i]) * p.scale_log2;
                    }
                }
                tc_fence_before();
                mbar_arrive(&bars.s_free);

                // send my partial scores (fp16) into the peer's receive buffer j&1
                const int kb = j & 1;
                if (j >= 2 && !warp_wait_cluster(&bars.send_credit[kb], ((j >> 1) - 1) & 1, deadline)) {
                    ok = false;
                    break;
                }
                const uint32_t dst = recv_peer + kb * RECV + h * 128;
#pragma unroll
                for (int c = 0; c < 8; ++c)
                    st_cluster_v4(dst + ((c ^ (h & 7)) << 4), pack_f16_sat(xc[8 * c], xc[8 * c + 1]),
                                  pack_f16_sat(xc[8 * c + 2], xc[8 * c + 3]), pack_f16_sat(xc[8 * c + 4], xc[8 * c + 5]),
                                  pack_f16_sat(xc[8 * c + 6], xc[8 * c + 7]));
                mbar_arrive_cluster(&bars.recv_full[kb], peer);
            }
            if (j >= 1) {
                const int jp = j - 1, kp = jp & 1;
                if (!warp_wait_cluster(&bars.recv_full[kp], (jp >> 1) & 1, deadline)) { ok = false; break; }
                {
                    const uint32_t src = recv_local + kp * RECV + h * 128;
#pragma unroll
                    for (int c = 0; c < 8; ++c) {
                        uint32_t a0, a1, a2, a3;
                        asm volatile("ld.shared.v4.b32 {%0,%1,%2,%3}, [%4];"
                                     : "=r"(a0), "=r"(a1), "=r"(a2), "=r"(a3)
                                     : "r"(src + ((c ^ (h & 7)) << 4)));
                        const float2 f0 = unpack_f16(a0), f1 = unpack_f16(a1), f2 = unpack_f16(a2), f3 = unpack_f16(a3);
                        xp[8 * c] += f0.x, xp[8 * c + 1] += f0.y, xp[8 * c + 2] += f1.x, xp[8 * c + 3] += f1.y;
                        xp[8 * c + 4] += f2.x, xp[8 * c + 5] += f2.y, xp[8 * c + 6] += f3.x, xp[8 * c + 7] += f3.y;
                    }
                    mbar_arrive_cluster(&bars.send_credit[kp], peer);   // the peer may refill this buffer
                }

                // online softmax over block jp (lazy maximum)
                float bm = -INFINITY;
#pragma unroll
                for (int i = 0; i < NK; ++i) {
                    const bool valid = ((i & 1) ? (vpo >> (i >> 1)) : (vpe >> (i >> 1))) & 1u;
                    xp[i] = valid ? xp[i] : -INFINITY;
                    bm = fmaxf(bm, xp[i]);
                }
                float f = 1.f;
                if (bm > m + RESCALE_T) {
                    f = ex2(m - bm);   // m = -inf -> 0
                    m = bm;
                }
                uint32_t pk[NK / 2];
                float sum = 0.f;
#pragma unroll
                for (int i = 0; i < NK; i += 2) {
                    const float p0 = ex2(xp[i] - m), p1 = ex2(xp[i + 1] - m);   // -inf -> 0
                    sum += p0 + p1;
                    pk[i / 2] = pack_bf16(p0, p1);
                }
                if (m == -INFINITY) {   // nothing valid so far: P must be zero, not NaN
                    sum = 0.f;
#pragma unroll
                    for (int i = 0; i < NK / 2; ++i) pk[i] = 0u;
                }
                l = l * f + sum;

                // P and O are in use by PV(jp-1) until it completes
                if (jp > 0) {
                    if (!warp_wait(&bars.pv_done, (jp - 1) & 1, deadline)) { ok = false; break; }
                    tc_fence_after();
                    if (__any_sync(0xffffffffu, f != 1.f)) {
#pragma unroll 1
                        for (int c0 = 0; c0 < 256; c0 += 16) {
                            uint32_t v[16];
                            tmem_ld16(trow + O_COL + c0, v);
                            tmem_ld_wait();
#pragma unroll
                            for (int i = 0; i < 16; ++i) v[i] = __float_as_uint(__uint_as_float(v[i]) * f);
                            tmem_st16(trow + O_COL + c0, v);
                        }
                    }
                }
                {
                    uint32_t v[16];
#pragma unroll
                    for (int i = 0; i < 16; ++i) v[i] = pk[i];
                    tmem_st16(trow + P_COL, v);
#pragma unroll
                    for (int i = 0; i < 16; ++i) v[i] = pk[16 + i];
                    tmem_st16(trow + P_COL + 16, v);
                }
                tmem_st_wait();
                tc_fence_before();
                mbar_arrive(&bars.p_full);
            }
#pragma unroll
            for (int i = 0; i < NK; ++i) xp[i] = xc[i];
            vpe = vce;
            vpo = vco;
        }
        if (ok && nblk > 0) {
            if (!warp_wait(&bars.pv_done, (nblk - 1) & 1, deadline)) ok = false;
            tc_fence_after();
        }
        if (!ok) fail(p);

        // ------------------------------------------------------------ epilogue
        const bool have = ok && nblk > 0 && l > 0.f;
        const float inv = have ? 1.f / l : 0.f;
        float *dst = p.n_split == 1 ? p.o_out + ((size_t)b * H + h) * C + 256 * r
                                    : p.part_o + ((size_t)unit * H + h) * C + 256 * r;
#pragma unroll 1
        for (int c0 = 0; c0 < 256; c0 += 16) {
            float4 o4[4];
            if (have) {
                uint32_t v[16];
                tmem_ld16(trow + O_COL + c0, v);
                tmem_ld_wait();
#pragma unroll
                for (int q = 0; q < 4; ++q)
                    o4[q] = make_float4(__uint_as_float(v[4 * q]) * inv, __uint_as_float(v[4 * q + 1]) * inv,
                                        __uint_as_float(v[4 * q + 2]) * inv, __uint_as_float(v[4 * q + 3]) * inv);
            } else {
#pragma unroll
                for (int q = 0; q < 4; ++q) o4[q] = make_float4(0.f, 0.f, 0.f, 0.f);
            }
#pragma unroll
            for (int q = 0; q < 4; ++q) reinterpret_cast<float4 *>(dst + c0)[q] = o4[q];
        }
        if (p.n_split > 1)
            p.part_lse[((size_t)unit * 2 + r) * H + h] = have ? m + __log2f(l) : -INFINITY;
    }

    tc_fence_before();
    __syncthreads();
    if (warp == MMA_WARP) {
        tc_fence_after();
        tmem_dealloc(tmem, TMEM_COLS);
    }
    cluster_sync();   // the peer no longer writes into this CTA's shared memory
}

// grid (B, H), 128 threads x 4 columns: merge the splits of one (sequence,
// head); each latent half uses the masses its own CTA computed.
__global__ void __launch_bounds__(128) combine_kernel(const float *__restrict__ part_o,
                                                      const float *__restrict__ part_lse, int n_split,
                                                      float *__restrict__ o_out) {
    const int b = blockIdx.x, h = blockIdx.y, c = threadIdx.x * 4, half = c >= 256 ? 1 : 0;
    float M = -INFINITY;
    for (int s = 0; s < n_split; ++s) M = fmaxf(M, part_lse[(((size_t)b * n_split + s) * 2 + half) * H + h]);
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    float L = 0.f;
    if (M != -INFINITY) {
        for (int s = 0; s < n_split; ++s) {
            const size_t u = (size_t)b * n_split + s;
            const float lse = part_lse[(u * 2 + half) * H + h];
            if (lse == -INFINITY) continue;
            const float w = exp2f(lse - M);
            L += w;
            const float4 v = *reinterpret_cast<const float4 *>(part_o + (u * H + h) * C + c);
            acc.x = fmaf(w, v.x, acc.x), acc.y = fmaf(w, v.y, acc.y);
            acc.z = fmaf(w, v.z, acc.z), acc.w = fmaf(w, v.w, acc.w);
        }
    }
    const float inv = L > 0.f ? 1.f / L : 0.f;
    *reinterpret_cast<float4 *>(o_out + ((size_t)b * H + h) * C + c) =
        make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
}

}  // namespace attn

// ------------------------------------------------------------------ host side
int attn_n_split(int B, int K) {
    const int pairs = 74;   // 148 SMs, one CTA pair per unit
    int n = B >= pairs ? 1 : pairs / B;
    const int max_split = (K + 127) / 128;
    if (n > max_split) n = max_split;
    return n < 1 ? 1 : n;
}

size_t attn_workspace(int B, int K, int *n_split_out, int *split_len_out) {
    int n = attn_n_split(B, K);
    int len = (K + n - 1) / n;
    len = (len + attn::NK - 1) / attn::NK * attn::NK;
    n = (K + len - 1) / len;
    if (n_split_out) *n_split_out = n;
    if (split_len_out) *split_len_out = len;
    if (n == 1) return 0;
    const size_t units = (size_t)B * n;
    return units * H * C * sizeof(float) + units * 2 * H * sizeof(float);
}

int launch_attn(const uint16_t *q_lat, const uint16_t *kv, const uint16_t *pe, int S_cap, const int32_t *topk, int K,
                const int32_t *end_pos, int B, float softmax_scale, float *o_out, void *ws, int32_t *status,
                cudaStream_t s, int *launches) {
    int n_split = 1, split_len = K;
    attn_workspace(B, K, &n_split, &split_len);
    attn::Params p{};
    p.q_lat = q_lat;
    p.kv = kv;
    p.pe = pe;
    p.topk = topk;
    p.end_pos = end_pos;
    p.S_cap = S_cap;
    p.K = K;
    p.B = B;
    p.scale_log2 = softmax_scale * 1.4426950408889634f;
    p.n_split = n_split;
    p.split_len = split_len;
    p.status = status;
    if (n_split == 1) {
        p.o_out = o_out;
    } else {
        const size_t units = (size_t)B * n_split;
        p.part_o = static_cast<float *>(ws);
        p.part_lse = p.part_o + units * H * C;
    }
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return MLA_ERR_CUDA;
    static bool attr_set[64] = {};
    if (dev < 0 || dev >= 64 || !attr_set[dev]) {
        if (cudaFuncSetAttribute(attn::attn_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, attn::SMEM_BYTES) !=
            cudaSuccess)
            return MLA_ERR_CUDA;
        if (dev >= 0 && dev < 64) attr_set[dev] = true;
    }
    const ProfileHook &hook = profile_hook();
    const bool timed = hook.start && hook.stop;
    if (timed && cudaEventRecord(hook.start, s) != cudaSuccess) return MLA_ERR_CUDA;
    attn::attn_kernel<<<2 * B * n_split, attn::THREADS, attn::SMEM_BYTES, s>>>(p);
    if (cudaGetLastError() != cudaSuccess) return MLA_ERR_CUDA;
    if (timed && cudaEventRecord(hook.stop, s) != cudaSuccess) return MLA_ERR_CUDA;
    int n = 1;
    if (n_split > 1) {
        attn::combine_kernel<<<dim3(B, H), 128, 0, s>>>(p.part_o, p.part_lse, n_split, o_out);
        if (cudaGetLastError() != cudaSuccess) return MLA_ERR_CUDA;
        ++n;
    }
    if (launches) *launches += n;
    return MLA_OK;
}

}  // namespace mla
