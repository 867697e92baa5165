// Sparse latent attention on the 5th-generation tensor cores (tcgen05 + TMEM),
// fed by 16-byte cp.async row gathers from eight warps.
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
//   QK  : S_r[128 heads, 64 keys] = Q_r . K_r^T, 16 MMAs of K=16 with the
//         latent part of Q_r in TMEM and 2 with its rotary part in shared
//         memory; B = the gathered tile, K-major.
//   The two partial score tiles are exchanged through distributed shared
//   memory and summed: each softmax warp writes its 32 heads' raw scores as
//   fp16 into its quarter of a send buffer and ships that 4 KB quarter with
//   its own bulk copy into a ring of three receive buffers in the peer, where
//   one mbarrier per quarter counts the arriving bytes, so a warp waits only
//   for its own heads' half of the scores.  Both CTAs then hold the full
//   scores and run the same online softmax.
//   PV  : O_r[128 heads, 256 latent] += P[128, 64] . V_r[64, 256]  (A = P
//         as bf16 in shared memory, B = the same gathered tile read MN-major).
// TMEM per CTA: O_r columns [0,256), latent Q_r [256,384), two score
// buffers S0 [384,448) and S1 [448,512).  A score buffer is released as soon
// as the softmax has read it; P(j) is written (128-byte-swizzled, K-major)
// over the peer's partial scores in receive slot j mod 3, row by row by the
// thread that consumed that row.
//
// Warp roles (640 threads, five warpgroups):
//   warps 0-7   gather: every thread copies 9 of a block's 2304 16-byte
//               chunks with cp.async; the stage's mbarrier is signalled by
//               the copies' completion (cp.async.mbarrier.arrive.noinc), so
//               a block is published as soon as its own bytes have landed;
//   warp 8      issues QK(j) once stage j is full and score buffer j%2 has
//               been read (block j-2);
//   warp 9      issues PV(j) once P(j) is in shared memory;
//   warp 11     forwards each completed PV(j) to the peer as a ring credit
//               (warp 10 is idle);
//   warps 12-15 softmax of the even blocks, warps 16-19 of the odd blocks
//               (ping-pong): one thread per head, all 64 keys of its block;
//               before the first block, one of their threads loads Q_r by
//               TMA (the latent part through gather stages 2-3, whose first
//               blocks wait for it, the rotary part into its place) and the
//               warpgroups move its latent part into TMEM.
// The selection of the unit is staged in shared memory once (positions
// outside [0, end_pos) become -1), so no global index load sits on the
// per-block path: as 32-bit positions (up to 2048 entries per unit), or as
// 16-bit ones when a unit holds more (up to 4096, which the split policy
// allows only over caches of at most 65,535 rows); longer selections are
// split across units.  A unit processes its blocks up to the one that holds
// its last position: blocks of padding alone after it (a selection row
// wider than the cached positions, early in a sequence) would add nothing.
//
// Online softmax with a lazy running maximum m (log2 units): block j's
// maximum replaces m only when it exceeds m by more than 8, which keeps
// every exponent <= 2^8; numerator and denominator share m, so the result is
// exact up to rounding.  m passes from the warpgroup of block j-1 to that of
// block j through shared memory (one value per head); whichever warpgroup
// raises m rescales O (after PV(j-1)), and each keeps its own running sum,
// brought to the current m when it sees m change.
//
// Softmax warpgroups take blocks in turn (NWG of them; two, the measured
// best: three with four gather warps ran slower).  Every barrier a warpgroup
// waits on for its own blocks is indexed by the block's warpgroup (j % NWG,
// phase j / NWG), so each waiter sees the phases of its barrier strictly in
// order.
//
// Exchange ring with direct credits: block i (i >= 3) is sent into the
// peer's slot i mod 3 only after the peer's PV(i-3) has read P(i-3) from that
// slot -- the peer's credit warp (warp 11) waits for each of its PVs and
// arrives on this CTA's credit barrier of the slot.  The peer's copy of block
// i then lands here after this CTA's own PV(i-3), and so after its softmax of
// block i-3 has passed that slot's previous receive phase.  The warp of block
// i that owns a quarter posts that quarter's receive byte count after the
// copy of block i-1's same quarter has read the send buffer, i.e. after the
// other warpgroup's warp of that quarter finished block i-3.  Each CTA runs at
// most three blocks ahead of the other.  The issuer lanes (QK, PV, credits)
// poll their barriers rather than suspend: they have nothing else to do, and
// the QK issuer's reaction to a landed stage is on every block's path.
#include "common.cuh"
#include "kernels.cuh"
#include "tc05.cuh"

#include <math.h>

namespace mla {
namespace attn {

using namespace tc;

constexpr int NK = 64;                       // keys per block
constexpr int NS = 4;                        // gather pipeline stages
constexpr int STAGE_KV = 4 * NK * 128;       // 4 atom columns of 64 latent x 64 keys (128B swizzle)
constexpr int STAGE_PE = NK * 64;            // 32 rotary columns x 64 keys (64B swizzle)
constexpr int STAGE = STAGE_KV + STAGE_PE;   // 36864
constexpr int NRECV = 3;                     // exchange ring depth
constexpr int RECV = H * NK * 2;             // fp16 partial scores of the peer, 128 x 64
constexpr int IDX_BYTES = 8192;              // the unit's selection, staged in shared memory
constexpr int IDX_CAP = IDX_BYTES / 4;       // entries as 32-bit positions
constexpr int IDX_CAP16 = IDX_BYTES / 2;     // entries as 16-bit positions (caches of at most 65,535 rows)
constexpr int QROPE = H * 64;                // rotary part of Q_r: 128 heads x 32 bf16 (64B swizzle)
constexpr int SEND = RECV;                   // this CTA's partial scores of one block, shipped by bulk copy
constexpr int QUARTER = RECV / 4;            // one warp's 32 rows of a block's scores, its own bulk copy
constexpr int Q_STAGE = 2;                   // Q_r's latent part arrives by TMA in gather stages 2 and 3
constexpr int QBOX = 64 * H * 2;             // one 128B-swizzled box of Q_r: 64 latent columns x 128 heads
static_assert((NS - Q_STAGE) * STAGE >= 4 * QBOX && (Q_STAGE * STAGE) % 1024 == 0, "Q_r staging in the gather stages");
constexpr int SMEM_BYTES = NS * STAGE + NRECV * RECV + QROPE + IDX_BYTES + SEND + 1024;
constexpr uint32_t O_COL = 0, Q_COL = 256, S_COL = 384, TMEM_COLS = 512;   // S buffer k at S_COL + 64 k
constexpr int THREADS = 640;                 // 20 warps
constexpr int NWG = 2;                       // softmax warpgroups, taking blocks in turn
constexpr int GATHER_WARPS = 16 - 4 * NWG;   // the rest of the 20 warps, after the MMA warpgroup
constexpr int GATHER_THREADS = 32 * GATHER_WARPS;
constexpr int CPT = NK * 36 / GATHER_THREADS;   // 16-byte chunks per gather thread per block
static_assert(CPT * GATHER_THREADS == NK * 36, "chunks must divide evenly");
constexpr int QK_WARP = GATHER_WARPS, PV_WARP = GATHER_WARPS + 1;
constexpr int CREDIT_WARP = GATHER_WARPS + 3;
constexpr int SOFTMAX_WARP0 = GATHER_WARPS + 4;
constexpr int WG_THREADS = 128;
static_assert(NRECV == NWG || NWG == 2, "with three warpgroups each owns one receive slot");
// registers per thread after reallocation, within the launch's 640 x 96
constexpr int REG_GATHER = NWG == 3 ? 80 : 72, REG_MMA = NWG == 3 ? 40 : 56, REG_SOFTMAX = NWG == 3 ? 120 : 136;
static_assert(GATHER_THREADS * REG_GATHER + 128 * REG_MMA + NWG * WG_THREADS * REG_SOFTMAX <= THREADS * 96,
              "register split");
// latent columns of O_r that warpgroup w normalises and writes: [ocol(w), ocol(w+1))
__host__ __device__ constexpr int ocol(int w) { return 16 * ((16 * w) / NWG); }
// fp32 staging pitch of warpgroup w's part of a row: its 16-byte chunks rounded up to whole swizzle groups of 8
__host__ __device__ constexpr int stage_row_bytes(int w) { return ((((ocol(w + 1) - ocol(w)) * 4 / 16) + 7) / 8) * 8 * 16; }
constexpr float RESCALE_T = 8.f;             // lazy-max threshold (log2 units)
constexpr float SCORE_RANGE = 2048.f;        // largest partial score sent without MLA_DEV_SCORE_RANGE

struct Params {
    const uint16_t *q_lat;
    const uint16_t *kv;
    const uint16_t *pe;
    const int32_t *topk;
    const int32_t *end_pos;
    int S_cap, K, B;    // B: query rows, T per sequence (row b is token b % T of sequence b / T)
    int T;
    float scale_log2;   // softmax_scale * log2(e)
    int n_split, split_len;   // split_len <= IDX_CAP (32-bit staging) or IDX_CAP16 (16-bit)
    float *o_out;       // n_split == 1: normalised o, fp32 [B][128][512] (or NULL)
    uint16_t *o_b16;    // n_split == 1: normalised o, bf16 [B][128][512] (or NULL)
    float *part_o;      // n_split > 1: per-split normalised o, fp32 [B*n_split][128][512]
    uint16_t *part_o16; // n_split > 1 instead of part_o, when the up-projection merges the splits:
                        // the same partials as bf16 (its operand is bf16 anyway)
    float *part_lse;    // n_split > 1: log2 of the split's softmax mass, [B*n_split][2][128]
    int32_t *status;
    uint64_t wait_ns;   // limit of every bounded wait
};

struct Bars {
    uint64_t full[NS], empty[NS];
    // Barriers a warpgroup waits on for its own blocks are kept per warpgroup
    // (index j % NWG, phase j / NWG): a warpgroup then waits every phase of
    // its barrier in order, and a parity wait can never refer to a phase two
    // behind or ahead.  s_free is waited by the QK issuer alone, in order.
    uint64_t s_full[NWG], pv_done[NWG], s_free[2], q_ready;
    uint64_t q_full;       // Q_r has landed (TMA): latent part in stages 2-3, rotary part in place
    uint64_t p_full[NWG];  // P of warpgroup w's blocks (one barrier per warpgroup: with three, the
                           // warpgroups of blocks j and j+2 differ and must not share a phase)
    uint64_t recv_full[NRECV][4];   // quarter q (heads 32q .. 32q+31) of the peer's block in slot k
    uint64_t credit[NRECV];   // the peer's PV(i) has read P(i) from its slot i mod 3 (phase i / 3), so
                              // block i + 3 may be sent into it; arrived on by the peer's credit warp
    uint64_t m_ready[NWG]; // m after block j is in mval[j % 2] (phase j / NWG of m_ready[j % NWG])
    uint64_t l_ready;      // both running sums are in lsum (the send buffer, after the last copy)
    uint64_t drain[2];     // MMA issuers (QK, PV): every MMA they issued has completed
    int send_done[4];      // copies 0 .. send_done[q]-1 of quarter q have read it from the send
                           // buffer (a counter, not a barrier: the warp of block j waits for the
                           // copy of block j-1 without having seen the copy of block j-2 complete)
    uint32_t tmem_base;
    int last_valid[THREADS / 32];   // per warp: the last staged entry that holds a position (-1: none)
    int nblk;                       // blocks the unit processes (up to the one holding its last position)
    float mval[2][H];
};

__device__ __forceinline__ void fail(const Params &p) { report(p.status, MLA_DEV_TIMEOUT); }

// blocks the unit processes, as published in shared memory before the cluster barrier
__device__ __forceinline__ int unit_blocks(const Bars &bars) { return *reinterpret_cast<const volatile int *>(&bars.nblk); }

// Entry i of the staged selection: a position, or -1 for padding and positions
// outside the row's visible range.  IDX16: 16-bit positions, 0xFFFF for none
// (units of more than IDX_CAP entries, over caches of at most 65,535 rows).
template <bool IDX16>
__device__ __forceinline__ int sel_at(const int32_t *sidx, int i) {
    if constexpr (IDX16) {
        const uint32_t v = reinterpret_cast<const uint16_t *>(sidx)[i];
        return v == 0xFFFFu ? -1 : int(v);
    } else {
        return sidx[i];
    }
}

// Bounded wait until a shared-memory counter written by another thread of the
// CTA reaches `target` (warp-uniform result).
__device__ __forceinline__ bool wait_count(const int *counter, int target, const Deadline &deadline) {
    bool ok = true;
    for (uint32_t i = 0; *reinterpret_cast<const volatile int *>(counter) < target; ++i) {
        if (i >= 2) __nanosleep(32);
        if ((i & 31) == 31 && globaltimer_ns() > deadline.t) {
            ok = false;
            break;
        }
    }
    __threadfence_block();
    return __all_sync(0xffffffffu, ok);
}

// warp-uniform bounded waits: every lane of the warp takes the same branch afterwards
__device__ __forceinline__ bool warp_wait(uint64_t *bar, uint32_t parity, const Deadline &deadline) {
    return __all_sync(0xffffffffu, wait_until(bar, parity, deadline));
}

// Bounded wait that polls without suspending: for the single-lane issuer
// warps, which have nothing else to do and must act as soon as a phase completes.
__device__ __forceinline__ bool wait_spin(uint64_t *bar, uint32_t parity, const Deadline &d) {
#pragma unroll 1
    for (uint32_t i = 0;; ++i) {
        if (mbar_test(bar, parity)) return true;
        if ((i & 63) == 63 && globaltimer_ns() > d.t) return false;
    }
}
// maximum of three (PTX max.f32 with three sources, sm_100 and later)
__device__ __forceinline__ float fmax3(float a, float b, float c) {
    float r;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
    return r;
}
// lo_acc += the low fp16 half of w, hi_acc += the high half: PTX's mixed-precision
// add widens the half exactly and rounds once, as a conversion and an fp32 add would
__device__ __forceinline__ void add_f16x2(uint32_t w, float &lo_acc, float &hi_acc) {
    asm("{\n .reg .f16 lo, hi;\n mov.b32 {lo, hi}, %2;\n add.rn.f32.f16 %0, lo, %0;\n add.rn.f32.f16 %1, hi, %1;\n}"
        : "+f"(lo_acc), "+f"(hi_acc) : "r"(w));
}


template <bool IDX16>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(THREADS, 1)
    attn_kernel(const __grid_constant__ CUtensorMap qmap, const __grid_constant__ CUtensorMap qrmap, Params p) {
    extern __shared__ uint8_t smem_raw[];
    __shared__ Bars bars;
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *stages = smem;
    uint8_t *recv = smem + NS * STAGE;
    uint8_t *qrope = recv + NRECV * RECV;
    int32_t *sidx = reinterpret_cast<int32_t *>(qrope + QROPE);
    uint8_t *sendbuf = qrope + QROPE + IDX_BYTES;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const uint32_t r = cluster_rank(), peer = r ^ 1u;
    // Launched as a programmatic dependent of the preceding grid (the query
    // absorption): the caches, the selection and end_pos are inputs of the
    // step, so the selection is staged and the gather starts at once; q_lat,
    // which that grid writes, is read only by the softmax warpgroups, after
    // their griddepcontrol.wait.
    const int unit = blockIdx.x >> 1;
    const int b = unit / p.n_split, split = unit % p.n_split;   // query row
    const int cb = b / p.T;                                     // its sequence in the caches
    const int e_seq = p.end_pos[cb];
    const bool seq_ok = e_seq >= p.T && e_seq <= p.S_cap;
    // keys [0, e) are visible to the row: the selection merged with the causal mask
    const int e = e_seq - p.T + (b - cb * p.T) + 1;
    const int t0 = split * p.split_len;
    const int t1 = min(p.K, t0 + p.split_len);
    // blocks of the unit's selection: their loads do not wait for end_pos (a bad end_pos
    // leaves every entry invalid and the unit empty), so the two latencies overlap
    const int nblk_sel = t1 > t0 ? (t1 - t0 + NK - 1) / NK : 0;
    if (!seq_ok && tid == 0 && r == 0 && split == 0) report(p.status, MLA_DEV_BAD_END_POS);

    // the unit's selection, padded to whole blocks; padding and positions
    // outside [0, end_pos) become -1 (four independent loads per thread)
    {
        const int32_t *sel = p.topk + (size_t)b * p.K;
        const int n = nblk_sel * NK;
        int last = -1;
        for (int i0 = tid; i0 < n; i0 += 4 * THREADS) {
            int id[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int i = i0 + u * THREADS, slot = t0 + i;
                id[u] = (i < n && slot < t1) ? sel[slot] : -1;
            }
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int i = i0 + u * THREADS;
                if (i < n) {
                    const bool valid = seq_ok && id[u] >= 0 && id[u] < e;
                    if (valid) last = i;
                    if constexpr (IDX16)
                        reinterpret_cast<uint16_t *>(sidx)[i] = valid ? uint16_t(id[u]) : uint16_t(0xFFFFu);
                    else
                        sidx[i] = valid ? id[u] : -1;
                }
            }
        }
        // the unit's blocks end with the one that holds its last position: blocks of
        // padding alone after it are not processed (they would add nothing)
#pragma unroll
        for (int off = 16; off; off >>= 1) last = max(last, __shfl_xor_sync(0xffffffffu, last, off));
        if (lane == 0) bars.last_valid[warp] = last;
    }
    if (tid == 0) {
        for (int s = 0; s < NS; ++s) mbar_init(&bars.full[s], GATHER_THREADS), mbar_init(&bars.empty[s], 1);
        for (int k = 0; k < 2; ++k) {
            mbar_init(&bars.s_free[k], WG_THREADS);
        }
        for (int k = 0; k < NWG; ++k) {
            mbar_init(&bars.p_full[k], WG_THREADS);
            mbar_init(&bars.s_full[k], 1);
            mbar_init(&bars.pv_done[k], 1);
            mbar_init(&bars.m_ready[k], WG_THREADS);
        }
        mbar_init(&bars.q_ready, NWG * WG_THREADS);
        mbar_init(&bars.q_full, 1);
        mbar_init(&bars.l_ready, NWG * WG_THREADS);
        mbar_init(&bars.drain[0], 1);
        mbar_init(&bars.drain[1], 1);
        for (int q = 0; q < 4; ++q) bars.send_done[q] = 0;
        for (int k = 0; k < NRECV; ++k) {
            for (int q = 0; q < 4; ++q) mbar_init(&bars.recv_full[k][q], 1);
            mbar_init(&bars.credit[k], 1);
        }
        fence_mbar_init();
    }
    if (warp == QK_WARP) {
        tmem_alloc(&bars.tmem_base, TMEM_COLS);
        tmem_relinquish();
    }
    __syncthreads();   // every warp's last staged position is in
    if (tid == 0) {
        // blocks to process (both CTAs of the pair stage the same selection and agree)
        int last = -1;
        for (int v = 0; v < THREADS / 32; ++v) last = max(last, bars.last_valid[v]);
        bars.nblk = (last + NK) / NK;
    }
    tc_fence_before();
    cluster_sync();   // barriers of both CTAs initialised, TMEM address published, selection staged
    tc_fence_after();
    // the block count is read where it is used (from shared memory) rather than
    // held in a register across the whole kernel
    const uint32_t tmem = bars.tmem_base;
    const Deadline deadline = make_deadline(p.wait_ns);

    if (warp < GATHER_WARPS) {
        // ------------------------------------------------------------ gather producers
        // Chunk ch = tid + GATHER_THREADS q (q < CPT) of a block belongs to key ch / 36;
        // chunks 0..31 of a key are its latent half (4 atom columns x 8,
        // 128-byte swizzle), 32..35 its rotary half (64-byte swizzle).
        // Unselected keys are zero-filled.
        regs_dec<REG_GATHER>();
        uint32_t dst_off[CPT];
        int src_off[CPT], key[CPT];
        uint32_t pe_mask = 0;
#pragma unroll
        for (int q = 0; q < CPT; ++q) {
            const int ch = tid + GATHER_THREADS * q;
            key[q] = ch / 36;
            const int c = ch % 36;
            if (c < 32) {
                const int a = c >> 3, cc = c & 7;
                dst_off[q] = a * (NK * 128) + sw128(key[q], cc);
                src_off[q] = 256 * r + 64 * a + 8 * cc;
            } else {
                const int cc = c - 32;
                dst_off[q] = STAGE_KV + sw64(key[q], cc);
                src_off[q] = 32 * r + 8 * cc;
                pe_mask |= 1u << q;
            }
        }
        const uint16_t *kvb = p.kv + (size_t)cb * p.S_cap * C;
        const uint16_t *peb = p.pe + (size_t)cb * p.S_cap * DR;
        for (int j = 0; j < unit_blocks(bars); ++j) {
            const int s = j % NS;
            if (j >= NS && !warp_wait(&bars.empty[s], ((j / NS) - 1) & 1, deadline)) {
                fail(p);
                break;
            }
            // stages 2 and 3 first hold Q_r's latent part: their first blocks wait
            // until the softmax warpgroups have moved it into TMEM
            if (j >= Q_STAGE && j < NS && !warp_wait(&bars.q_ready, 0, deadline)) {
                fail(p);
                break;
            }
            const uint32_t base = smem_u32(stages + s * STAGE);
            const int bofs = j * NK;
#pragma unroll
            for (int q = 0; q < CPT; ++q) {
                const int id = sel_at<IDX16>(sidx, bofs + key[q]);
                const size_t row = id < 0 ? 0 : (size_t)id;
                const uint16_t *src = ((pe_mask >> q) & 1u) ? peb + row * DR + src_off[q] : kvb + row * C + src_off[q];
                cp_async16(base + dst_off[q], src, id < 0 ? 0u : 16u);
            }
            // the stage's mbarrier counts this thread once its copies have landed
            cp_async_arrive_noinc(&bars.full[s]);
        }
        cp_async_wait<0>();   // no copy of this thread outlives the branch
    } else if (warp < SOFTMAX_WARP0) {
        // ------------------------------------------------------------ MMA issuers (warp 8: QK, warp 9: PV)
        regs_dec<REG_MMA>();
        if (lane == 0 && unit_blocks(bars) > 0 && (warp == QK_WARP || warp == PV_WARP)) {
            bool ok = true;
            if (warp == QK_WARP) {
                constexpr uint32_t idesc_qk = idesc_bf16(128, NK, false, false);
                ok = wait_until(&bars.q_ready, 0, deadline) && wait_until(&bars.q_full, 0, deadline);
                const uint32_t qr = smem_u32(qrope);
                for (int j = 0; ok && j < unit_blocks(bars); ++j) {
                    const int s = j % NS, k = j & 1;
                    // stage j gathered; score buffer k read by the softmax of block j-2
                    ok = wait_spin(&bars.full[s], (j / NS) & 1, deadline) &&
                         (j < 2 || wait_spin(&bars.s_free[k], ((j - 2) >> 1) & 1, deadline));
                    if (!ok) break;
                    // the stage was written by cp.async (generic proxy) and is read by the MMA (async proxy)
                    fence_proxy_async_smem();
                    tc_fence_after();
                    const uint32_t base = smem_u32(stages + s * STAGE);
                    const uint32_t sc = tmem + S_COL + 64 * k;
#pragma unroll
                    for (int kk = 0; kk < 16; ++kk)
                        mma_ts(sc, tmem + Q_COL + kk * 8,
                               smem_desc(base + (kk >> 2) * (NK * 128) + (kk & 3) * 32, 16, 1024, 2), idesc_qk, kk > 0);
#pragma unroll
                    for (int kk = 0; kk < 2; ++kk)
                        mma_ss(sc, smem_desc(qr + kk * 32, 16, 512, 4), smem_desc(base + STAGE_KV + kk * 32, 16, 512, 4),
                               idesc_qk, 1);
                    mma_commit(&bars.s_full[j % NWG]);
                }
            } else {
                constexpr uint32_t idesc_pv = idesc_bf16(128, 256, false, true);
                for (int j = 0; ok && j < unit_blocks(bars); ++j) {
                    const int s = j % NS;
                    ok = wait_spin(&bars.p_full[j % NWG], (j / NWG) & 1, deadline);
                    if (!ok) break;
                    tc_fence_after();
                    const uint32_t base = smem_u32(stages + s * STAGE);
                    const uint32_t pa = smem_u32(recv + (j % NRECV) * RECV);   // P(j), K-major, 128B swizzle
#pragma unroll
                    for (int kk = 0; kk < NK / 16; ++kk)
                        mma_ss(tmem + O_COL, smem_desc(pa + kk * 32, 16, 1024, 2),
                               smem_desc(base + kk * 2048, NK * 128, 1024, 2), idesc_pv, (j > 0 || kk > 0) ? 1u : 0u);
                    mma_commit(&bars.pv_done[j % NWG]);
                    mma_commit(&bars.empty[s]);
                }
            }
            // The dependent grid (value up-projection or split combine) may be
            // scheduled once every CTA has issued its last QK: all of this CTA's
            // cache reads have landed by then, so the up-projection's weight loads
            // do not compete with the gather and the Q loads at the start (a CTA
            // with no blocks counts when it exits).  The dependent reads this
            // grid's output only after its own griddepcontrol.wait, which returns
            // once this grid -- and so the grid before it -- has completed.
            if (warp == QK_WARP) grid_dep_launch();
            if (!ok) fail(p);
            // drain: every MMA this thread issued has completed before TMEM is released
            mma_commit(&bars.drain[warp - QK_WARP]);
            if (!wait_until(&bars.drain[warp - QK_WARP], 0, globaltimer_ns() + DRAIN_NS)) fail(p);
        }
        if (lane == 0 && unit_blocks(bars) > 0 && warp == CREDIT_WARP) {
            // hands each completed PV(i) to the peer as the credit for its block i + 3
            for (int i = 0; i + NRECV < unit_blocks(bars); ++i) {
                if (!wait_spin(&bars.pv_done[i % NWG], (i / NWG) & 1, deadline)) {
                    fail(p);
                    break;
                }
                mbar_arrive_cluster(&bars.credit[i % NRECV], peer);
            }
        }
    } else {
        // ------------------------------------------------------------ softmax warpgroups (in turn)
        // warpgroup w handles blocks j = w, w+NWG, ...; thread = head h, all 64 keys
        regs_inc<REG_SOFTMAX>();
        const int w = (warp - SOFTMAX_WARP0) >> 2;
        const int quad = warp & 3;
        const int h = 32 * quad + lane;
        const int wtid = (warp - SOFTMAX_WARP0 - 4 * w) * 32 + lane;   // 0..127 within the warpgroup
        const uint32_t trow = tmem + (uint32_t(32 * quad) << 16);
        bool ok = true;
        // q_lat comes from the preceding grid, and an earlier grid may still read
        // the buffers the epilogue writes: both wait for it to complete
        grid_dep_wait();
        if (unit_blocks(bars) > 0) {
            // Q_r by TMA: the latent part [256r, 256r+256) as four 128B-swizzled boxes
            // of 64 columns x 128 heads into gather stages 2-3 (whose first blocks wait
            // for q_ready), the rotary part [512+32r, 512+32r+32) straight into its
            // place, K-major with the 64-byte swizzle.  Through the tensor memory
            // accelerator its 72 KB do not occupy the load path that the gather's
            // first cp.async wait for (per-thread loads of Q delayed the first block by
            // about 3.5 us).
            const uint32_t qst = smem_u32(stages + Q_STAGE * STAGE);
            if (w == 0 && wtid == 0) {
                mbar_expect_tx(&bars.q_full, 4 * QBOX + QROPE);
#pragma unroll
                for (int k = 0; k < 4; ++k) tma_load_2d(qst + k * QBOX, &qmap, 256 * r + 64 * k, b * H, &bars.q_full);
                tma_load_2d(smem_u32(qrope), &qrmap, C + 32 * r, b * H, &bars.q_full);
            }
            if (warp_wait(&bars.q_full, 0, deadline)) {
                // latent Q_r -> TMEM as 128 bf16 pairs per head: warpgroup w stores the
                // 16-column groups 8w/NWG .. 8(w+1)/NWG - 1 (group g = columns 32g ..
                // 32g+31, chunks 4(g&1) .. 4(g&1)+3 of box g/2)
                constexpr int QMAX = (8 + NWG - 1) / NWG;   // 16-column groups of a warpgroup, at most
                const int g0 = (8 * w) / NWG, ng = (8 * (w + 1)) / NWG - g0;
#pragma unroll
                for (int i = 0; i < QMAX; ++i) {
                    if (i >= ng) break;
                    const int g = g0 + i;
                    const uint32_t box = qst + (g >> 1) * QBOX;
                    uint32_t v[16];
#pragma unroll
                    for (int q = 0; q < 4; ++q)
                        asm volatile("ld.shared.v4.b32 {%0,%1,%2,%3}, [%4];"
                                     : "=r"(v[4 * q]), "=r"(v[4 * q + 1]), "=r"(v[4 * q + 2]), "=r"(v[4 * q + 3])
                                     : "r"(box + sw128(h, (g & 1) * 4 + q)));
                    tmem_st16(trow + Q_COL + 16 * g, v);
                }
                tmem_st_wait();
                tc_fence_before();
                mbar_arrive(&bars.q_ready);
            } else {
                ok = false;
                // the copies of Q_r may still be landing: wait for them (for at most the drain
                // limit) before warpgroup 1 stages its output in stages 2-3 or the CTA exits
                warp_wait(&bars.q_full, 0, make_deadline(DRAIN_NS));
            }
        }
        const uint32_t recv_local = smem_u32(recv);
        const uint32_t recv_peer = map_peer(recv_local, peer);
        const float sl2 = p.scale_log2;
        float m_mine = -INFINITY;   // m after this warpgroup's previous block
        float l = 0.f;              // this warpgroup's running sum, relative to m_mine
        for (int j = w; j < unit_blocks(bars) && ok; j += NWG) {
            const int k = j & 1;
            const uint32_t sc = trow + S_COL + 64 * k;
            // validity of the block's keys (bit i of vlo / vhi: key i / 32 + i)
            const uint32_t vlo = __ballot_sync(0xffffffffu, sel_at<IDX16>(sidx, j * NK + lane) >= 0);
            const uint32_t vhi = __ballot_sync(0xffffffffu, sel_at<IDX16>(sidx, j * NK + 32 + lane) >= 0);
            if (!warp_wait(&bars.s_full[w], (j / NWG) & 1, deadline)) { ok = false; break; }
            tc_fence_after();
            float x[64];
            {
                uint32_t v0[16], v1[16], v2[16], v3[16];
                tmem_ld16(sc, v0);
                tmem_ld16(sc + 16, v1);
                tmem_ld16(sc + 32, v2);
                tmem_ld16(sc + 48, v3);
                tmem_ld_wait();
                tc_fence_before();
                mbar_arrive(&bars.s_free[k]);   // QK(j+2) may overwrite the buffer
#pragma unroll
                for (int q = 0; q < 16; ++q) {
                    x[q] = __uint_as_float(v0[q]);
                    x[16 + q] = __uint_as_float(v1[q]);
                    x[32 + q] = __uint_as_float(v2[q]);
                    x[48 + q] = __uint_as_float(v3[q]);
                }
            }
            {
                // the partial scores travel to the peer as fp16, rounded to 11 significant
                // bits: flag magnitudes where that rounding reaches one unit of the raw score
                float a0 = 0.f, a1 = 0.f;
#pragma unroll
                for (int q = 0; q < 64; q += 4) {
                    a0 = fmax3(a0, fabsf(x[q]), fabsf(x[q + 1]));
                    a1 = fmax3(a1, fabsf(x[q + 2]), fabsf(x[q + 3]));
                }
                if (fmaxf(a0, a1) > SCORE_RANGE) report(p.status, MLA_DEV_SCORE_RANGE);
            }
            // ring credit: the peer's PV(j-3) has read P(j-3) from its slot j mod 3.  The
            // credit carries no data (the bulk copy that writes the slot is issued after
            // this wait has seen the phase), so a CTA-scope wait is enough.
            if (j >= NRECV && !warp_wait(&bars.credit[j % NRECV], ((j - NRECV) / NRECV) & 1, deadline)) {
                ok = false;
                break;
            }
            {
                const int kb = j % NRECV;
                // this warp's 32 rows of partial scores go to its quarter of the send buffer
                // (free once the copy of block j-1 -- the other warpgroup's warp of the same
                // quarter -- has read it), and lane 0 ships the quarter to the peer's slot
                if (!wait_count(&bars.send_done[quad], j, deadline)) { ok = false; break; }
                const uint32_t sb = smem_u32(sendbuf) + h * 128;
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                    const uint32_t a0 = pack_f16_sat(x[8 * c], x[8 * c + 1]), a1 = pack_f16_sat(x[8 * c + 2], x[8 * c + 3]);
                    const uint32_t a2 = pack_f16_sat(x[8 * c + 4], x[8 * c + 5]), a3 = pack_f16_sat(x[8 * c + 6], x[8 * c + 7]);
                    asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};" ::"r"(sb + ((c ^ (h & 7)) << 4)), "r"(a0), "r"(a1),
                                 "r"(a2), "r"(a3)
                                 : "memory");
                }
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) {
                    // the peer's quarter of block j arrives here: this warp announces its bytes
                    mbar_expect_tx(&bars.recv_full[kb][quad], QUARTER);
                    bulk_s2cluster(recv_peer + kb * RECV + quad * QUARTER, smem_u32(sendbuf) + quad * QUARTER,
                                   QUARTER, map_peer(smem_u32(&bars.recv_full[kb][quad]), peer));
                    bulk_commit();
                }
                if (!warp_wait(&bars.recv_full[kb][quad], (j / NRECV) & 1, deadline)) { ok = false; break; }
                if (lane == 0) {
                    // the copy has long read the quarter by now: hand it to the next block's warp
                    bulk_wait_read();
                    *reinterpret_cast<volatile int *>(&bars.send_done[quad]) = j + 1;
                }
                const uint32_t src = recv_local + kb * RECV + h * 128;
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                    uint32_t a0, a1, a2, a3;
                    asm volatile("ld.shared.v4.b32 {%0,%1,%2,%3}, [%4];"
                                 : "=r"(a0), "=r"(a1), "=r"(a2), "=r"(a3)
                                 : "r"(src + ((c ^ (h & 7)) << 4)));
                    add_f16x2(a0, x[8 * c], x[8 * c + 1]);
                    add_f16x2(a1, x[8 * c + 2], x[8 * c + 3]);
                    add_f16x2(a2, x[8 * c + 4], x[8 * c + 5]);
                    add_f16x2(a3, x[8 * c + 6], x[8 * c + 7]);
                }
            }
            if ((vlo & vhi) != 0xffffffffu) {
#pragma unroll
                for (int q = 0; q < 32; ++q) {
                    x[q] = ((vlo >> q) & 1u) ? x[q] : -INFINITY;
                    x[32 + q] = ((vhi >> q) & 1u) ? x[32 + q] : -INFINITY;
                }
            }
            float bm;
            {
                float t[22], u[8];
#pragma unroll
                for (int q = 0; q < 21; ++q) t[q] = fmax3(x[3 * q], x[3 * q + 1], x[3 * q + 2]);
                t[21] = x[63];
#pragma unroll
                for (int q = 0; q < 7; ++q) u[q] = fmax3(t[3 * q], t[3 * q + 1], t[3 * q + 2]);
                u[7] = t[21];
                bm = fmax3(fmax3(u[0], u[1], u[2]), fmax3(u[3], u[4], u[5]), fmaxf(u[6], u[7])) * sl2;   // log2 units
            }
            // running maximum: m after block j-1 comes from the other warpgroup
            float m_prev = -INFINITY;
            if (j >= 1) {
                if (!warp_wait(&bars.m_ready[(j - 1) % NWG], ((j - 1) / NWG) & 1, deadline)) { ok = false; break; }
                m_prev = bars.mval[(j - 1) & 1][h];
            }
            const float m = bm > m_prev + RESCALE_T ? bm : m_prev;
            bars.mval[k][h] = m;
            mbar_arrive(&bars.m_ready[w]);
            // bring this warpgroup's sum to m
            if (m != m_mine) {
                l = m_mine == -INFINITY ? 0.f : l * ex2(m_mine - m);
                m_mine = m;
            }
            uint32_t pk[32];
            float sum = 0.f;
            if (m == -INFINITY) {   // nothing valid so far: P must be zero, not NaN
#pragma unroll
                for (int q = 0; q < 32; ++q) pk[q] = 0u;
            } else {
                float s4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                for (int q = 0; q < 64; q += 2) {
                    const float p0 = ex2(fmaf(x[q], sl2, -m)), p1 = ex2(fmaf(x[q + 1], sl2, -m));   // -inf -> 0
                    s4[(q >> 1) & 3] += p0 + p1;
                    pk[q / 2] = pack_bf16(p0, p1);
                }
                sum = (s4[0] + s4[1]) + (s4[2] + s4[3]);
            }
            l += sum;
            // raising m rescales O, after PV(j-1) has added its block
            if (__any_sync(0xffffffffu, m != m_prev && m_prev != -INFINITY)) {
                const float f = (m != m_prev && m_prev != -INFINITY) ? ex2(m_prev - m) : 1.f;
                if (!warp_wait(&bars.pv_done[(j - 1) % NWG], ((j - 1) / NWG) & 1, deadline)) { ok = false; break; }
                tc_fence_after();
#pragma unroll 1
                for (int c0 = 0; c0 < 256; c0 += 16) {
                    uint32_t v[16];
                    tmem_ld16(trow + O_COL + c0, v);
                    tmem_ld_wait();
#pragma unroll
                    for (int q = 0; q < 16; ++q) v[q] = __float_as_uint(__uint_as_float(v[q]) * f);
                    tmem_st16(trow + O_COL + c0, v);
                }
            }
            // P(j) over this thread's row of receive slot j mod 3 (same swizzle as
            // the partial scores it replaces), then handed to the async proxy
            {
                const uint32_t prow = recv_local + (j % NRECV) * RECV + h * 128;
#pragma unroll
                for (int c = 0; c < 8; ++c)
                    asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};" ::"r"(prow + ((c ^ (h & 7)) << 4)),
                                 "r"(pk[4 * c]), "r"(pk[4 * c + 1]), "r"(pk[4 * c + 2]), "r"(pk[4 * c + 3])
                                 : "memory");
            }
            fence_proxy_async_smem();
            tc_fence_before();
            mbar_arrive(&bars.p_full[w]);
        }

        // drain: every copy this lane issued into the peer has been written before the
        // CTA reaches the final cluster barrier (after which the peer may exit)
        if (lane == 0) asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
        // ------------------------------------------------------------ final sums and epilogue
        // m after the last block; both sums are brought to it and added
        float m_fin = -INFINITY, lt = 0.f;
        if (ok && unit_blocks(bars) > 0) {
            const int jl = unit_blocks(bars) - 1;
            if (!warp_wait(&bars.m_ready[jl % NWG], (jl / NWG) & 1, deadline)) ok = false;
            if (ok) {
                m_fin = bars.mval[jl & 1][h];
                const float lw = (m_mine == -INFINITY || m_fin == -INFINITY) ? 0.f : l * ex2(m_mine - m_fin);
                // the sums go to the send buffer once the last copy has read it
                float *lsum = reinterpret_cast<float *>(sendbuf);   // 1 KB: quarter 0 of the buffer
                if (!wait_count(&bars.send_done[0], unit_blocks(bars), deadline)) ok = false;
                lsum[w * H + h] = lw;
                mbar_arrive(&bars.l_ready);
                if (!warp_wait(&bars.l_ready, 0, deadline)) ok = false;
                lt = 0.f;
#pragma unroll
                for (int v = 0; v < NWG; ++v) lt += lsum[v * H + h];
                if (ok && !warp_wait(&bars.pv_done[jl % NWG], (jl / NWG) & 1, deadline)) ok = false;
                tc_fence_after();
            }
        }
        if (!ok) fail(p);
        // warpgroup w normalises columns [ocol(w), ocol(w+1)) of O_r.  The rows
        // leave TMEM one head per thread; they are staged in shared memory (the
        // gather stages, idle once the last PV has completed) and then written
        // out by whole rows, so that every global store is coalesced.
        const bool tload = ok && unit_blocks(bars) > 0;   // warp-uniform: tcgen05.ld is warp-collective
        const bool have = tload && lt > 0.f;
        const float inv = have ? 1.f / lt : 0.f;
        const bool part16 = p.n_split > 1 && p.part_o16;
        const bool bf16_out = (p.n_split == 1 && p.o_b16) || part16;
        const int cw0 = ocol(w), ncol = ocol(w + 1) - cw0;
        const int esz = bf16_out ? 2 : 4;
        const int nch = ncol * esz / 16;                 // 16-byte chunks of this warpgroup's part of a row
        const int pitch_ch = (nch + 7) & ~7;             // staging row pitch in chunks (swizzle groups of 8)
        constexpr int STG_REGION = STAGE * NS / NWG;     // staging bytes per warpgroup
        static_assert(stage_row_bytes(NWG - 1) * H <= STG_REGION && stage_row_bytes(0) * H <= STG_REGION,
                      "the staged rows of a warpgroup fit in its share of the gather stages");
        const uint32_t stg = smem_u32(stages) + w * STG_REGION;
        const uint32_t srow = stg + h * pitch_ch * 16;
#pragma unroll 1
        for (int c0 = 0; c0 < ncol; c0 += 16) {
            uint32_t v0[16];
            if (tload) {
                tmem_ld16(trow + O_COL + cw0 + c0, v0);
                tmem_ld_wait();
            }
            float o[16];
#pragma unroll
            for (int q = 0; q < 16; ++q) o[q] = have ? __uint_as_float(v0[q]) * inv : 0.f;
            // chunk c of the row sits at (c & ~7) | ((c ^ h) & 7)
            if (bf16_out) {
#pragma unroll
                for (int i = 0; i < 2; ++i) {
                    const int c = c0 / 8 + i, pc = (c & ~7) | ((c ^ h) & 7);
                    asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};" ::"r"(srow + (pc << 4)),
                                 "r"(pack_bf16(o[8 * i], o[8 * i + 1])), "r"(pack_bf16(o[8 * i + 2], o[8 * i + 3])),
                                 "r"(pack_bf16(o[8 * i + 4], o[8 * i + 5])), "r"(pack_bf16(o[8 * i + 6], o[8 * i + 7]))
                                 : "memory");
                }
            } else {
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int c = c0 / 4 + i, pc = (c & ~7) | ((c ^ h) & 7);
                    asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};" ::"r"(srow + (pc << 4)),
                                 "f"(o[4 * i]), "f"(o[4 * i + 1]), "f"(o[4 * i + 2]), "f"(o[4 * i + 3])
                                 : "memory");
                }
            }
        }
        asm volatile("bar.sync %0, %1;" ::"r"(1 + w), "r"(WG_THREADS) : "memory");
        {
            const int col0 = 256 * r + cw0;
            const size_t row0 = p.n_split == 1 ? (size_t)b * H : (size_t)unit * H;
            uint8_t *dst = part16     ? reinterpret_cast<uint8_t *>(p.part_o16 + row0 * C + col0)
                           : bf16_out ? reinterpret_cast<uint8_t *>(p.o_b16 + row0 * C + col0)
                                      : reinterpret_cast<uint8_t *>((p.n_split == 1 ? p.o_out : p.part_o) + row0 * C + col0);
            const size_t pitch = bf16_out ? C * 2 : C * 4;   // bytes between the rows of two heads
#pragma unroll 4
            for (int idx = wtid; idx < H * nch; idx += WG_THREADS) {
                const int row = idx / nch, c = idx % nch, pc = (c & ~7) | ((c ^ row) & 7);
                uint32_t a0, a1, a2, a3;
                asm volatile("ld.shared.v4.b32 {%0,%1,%2,%3}, [%4];"
                             : "=r"(a0), "=r"(a1), "=r"(a2), "=r"(a3)
                             : "r"(stg + (row * pitch_ch + pc) * 16));
                *reinterpret_cast<uint4 *>(dst + row * pitch + c * 16) = make_uint4(a0, a1, a2, a3);
            }
        }
        if (p.n_split > 1 && w == 0)
            p.part_lse[((size_t)unit * 2 + r) * H + h] = have ? m_fin + __log2f(lt) : -INFINITY;
    }

    tc_fence_before();
    __syncthreads();
    if (warp == QK_WARP) {
        tc_fence_after();
        tmem_dealloc(tmem, TMEM_COLS);
    }
    cluster_sync();   // the peer no longer writes into this CTA's shared memory
}

// grid (B, H), 128 threads x 4 columns: merge the splits of one (sequence,
// head); each latent half uses the masses its own CTA computed.  Writes the
// normalised o as fp32 (o_out) or bf16 (o_b16), whichever is non-NULL.
__global__ void __launch_bounds__(128) combine_kernel(const float *__restrict__ part_o,
                                                      const float *__restrict__ part_lse, int n_split,
                                                      float *__restrict__ o_out, uint16_t *__restrict__ o_b16) {
    // the dependent grid (the up-projection) may start loading its weights now;
    // it reads this grid's output only after its own griddepcontrol.wait
    grid_dep_launch();
    grid_dep_wait();   // the partials come from the preceding attention grid
    const int b = blockIdx.x, h = blockIdx.y, c = threadIdx.x * 4, half = c >= 256 ? 1 : 0;
    float M = -INFINITY;
#pragma unroll 8
    for (int s = 0; s < n_split; ++s) M = fmaxf(M, part_lse[(((size_t)b * n_split + s) * 2 + half) * H + h]);
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    float L = 0.f;
    // an empty split has weight 0 and a zero o (its unit writes zeros): every split is
    // loaded unconditionally, so that the loads of several splits are in flight at once
#pragma unroll 8
    for (int s = 0; s < n_split; ++s) {
        const size_t u = (size_t)b * n_split + s;
        const float lse = part_lse[(u * 2 + half) * H + h];
        const float w = (M == -INFINITY || lse == -INFINITY) ? 0.f : exp2f(lse - M);
        L += w;
        const float4 v = *reinterpret_cast<const float4 *>(part_o + (u * H + h) * C + c);
        acc.x = fmaf(w, v.x, acc.x), acc.y = fmaf(w, v.y, acc.y);
        acc.z = fmaf(w, v.z, acc.z), acc.w = fmaf(w, v.w, acc.w);
    }
    const float inv = L > 0.f ? 1.f / L : 0.f;
    const size_t o = ((size_t)b * H + h) * C + c;
    if (o_b16)
        *reinterpret_cast<uint2 *>(o_b16 + o) = make_uint2(pack_bf16(acc.x * inv, acc.y * inv),
                                                           pack_bf16(acc.z * inv, acc.w * inv));
    else
        *reinterpret_cast<float4 *>(o_out + o) = make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
}

}  // namespace attn

// ------------------------------------------------------------------ host side
int attn_n_split(int B, int K, int S_cap) {
    const int pairs = 74;   // 148 SMs, one CTA pair per unit
    int n = B >= pairs ? 1 : pairs / B;
    // down to one 64-key block per unit: at P = 1,000, B = 1 (2048-wide rows) 32 units of one
    // block ran the kernel in 18.4 us against 20.4 us for 16 units of two
    const int max_split = (K + attn::NK - 1) / attn::NK;
    if (n > max_split) n = max_split;
    // a unit's selection fits in shared memory (16-bit positions when the cache allows)
    const int cap = S_cap <= 65535 ? attn::IDX_CAP16 : attn::IDX_CAP;
    const int min_split = (K + cap - 1) / cap;
    if (n < min_split) n = min_split;
    return n < 1 ? 1 : n;
}

size_t attn_workspace(int B, int K, int *n_split_out, int *split_len_out, int S_cap) {
    int n = attn_n_split(B, K, S_cap);
    int len = (K + n - 1) / n;
    len = (len + attn::NK - 1) / attn::NK * attn::NK;
    n = (K + len - 1) / len;
    if (n_split_out) *n_split_out = n;
    if (split_len_out) *split_len_out = len;
    if (n == 1) return 0;
    const size_t units = (size_t)B * n;
    return units * H * C * sizeof(float) + units * 2 * H * sizeof(float);
}

void attn_partials(int B, int K, int S_cap, void *ws, float **part_o, float **part_lse, int *n_split) {
    int n = 1, len = K;
    attn_workspace(B, K, &n, &len, S_cap);
    *n_split = n;
    const size_t units = (size_t)B * n;
    *part_o = n > 1 ? static_cast<float *>(ws) : nullptr;
    *part_lse = n > 1 ? static_cast<float *>(ws) + units * H * C : nullptr;
}

int launch_attn(const uint16_t *q_lat, const uint16_t *kv, const uint16_t *pe, int S_cap, const int32_t *topk, int K,
                const int32_t *end_pos, int B, int T, float softmax_scale, float *o_out, uint16_t *o_b16, void *ws,
                int32_t *status, cudaStream_t s, int *launches, bool merge_later) {
    int n_split = 1, split_len = K;
    attn_workspace(B, K, &n_split, &split_len, S_cap);
    attn::Params p{};
    p.q_lat = q_lat;
    p.kv = kv;
    p.pe = pe;
    p.topk = topk;
    p.end_pos = end_pos;
    p.S_cap = S_cap;
    p.K = K;
    p.B = B;
    p.T = T;
    p.scale_log2 = softmax_scale * 1.4426950408889634f;
    p.n_split = n_split;
    p.split_len = split_len;
    // 16-bit staging only where a unit holds more entries than 32-bit staging fits (the
    // split policy allows that only over caches of at most 65,535 rows)
    const bool idx16 = split_len > attn::IDX_CAP;
    p.status = status;
    p.wait_ns = wait_limit_ns();
    if (n_split == 1) {
        p.o_out = o_out;
        p.o_b16 = o_b16;
    } else {
        // the partials of a split the up-projection merges are written as bf16
        // (half the bytes each way); the combine kernel reads fp32 ones
        const size_t units = (size_t)B * n_split;
        if (merge_later)
            p.part_o16 = static_cast<uint16_t *>(ws);
        else
            p.part_o = static_cast<float *>(ws);
        p.part_lse = static_cast<float *>(ws) + units * H * C;
    }
    // Q_r of a unit arrives by TMA: q_lat viewed as [B*128 rows][576], boxes of
    // 64 latent columns (128B swizzle) and of the 32 rotary columns (64B swizzle)
    CUtensorMap qmap, qrmap;
    {
        const uint64_t dims[2] = {(uint64_t)QL, (uint64_t)B * H};
        const uint64_t strides[1] = {(uint64_t)QL * 2};
        const uint32_t box[2] = {64, H}, rbox[2] = {32, H};
        if (!make_tmap_bf16(&qmap, q_lat, 2, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B) ||
            !make_tmap_bf16(&qrmap, q_lat, 2, dims, strides, rbox, CU_TENSOR_MAP_SWIZZLE_64B))
            return MLA_ERR_CUDA;
    }
    static std::atomic<bool> smem_set[64];
    static std::atomic<bool> smem_set16[64];
    auto kern = idx16 ? attn::attn_kernel<true> : attn::attn_kernel<false>;
    if (!smem_attr_once(idx16 ? smem_set16 : smem_set, kern, attn::SMEM_BYTES)) return MLA_ERR_CUDA;
    const ProfileHook &hook = profile_hook();
    const bool timed = hook.start && hook.stop;
    // With the timing events in the stream the kernels are launched plainly:
    // an event between two grids would separate them anyway.
    if (timed && cudaEventRecord(hook.start, s) != cudaSuccess) return MLA_ERR_CUDA;
    if (launch_k(!timed, kern, dim3(2 * B * n_split), dim3(attn::THREADS), attn::SMEM_BYTES, s, qmap, qrmap, p) !=
        cudaSuccess)
        return MLA_ERR_CUDA;
    if (timed && cudaEventRecord(hook.stop, s) != cudaSuccess) return MLA_ERR_CUDA;
    int n = 1;
    if (n_split > 1 && !merge_later) {
        if (launch_k(!timed, attn::combine_kernel, dim3(B, H), dim3(128), 0, s, (const float *)p.part_o,
                     (const float *)p.part_lse, n_split, o_out, o_b16) != cudaSuccess)
            return MLA_ERR_CUDA;
        ++n;
    }
    if (launches) *launches += n;
    return MLA_OK;
}

}  // namespace mla
