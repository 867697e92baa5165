// Token-by-weight projections on either side of the attention:
//     Y[m][n] = sum_k X[m][k] * W[n][k]
// for a weight W [N][K] in the Linear layout and a handful of token rows
// X [M][K] (M = the decode batch), both bf16, fp32 accumulation.
//
// Source: DeepSeek-V3.2-Exp atlas, "Query heads" page, excerpt mla-init (the
// joint down-projection wkv_a = Linear(dim, 512 + 64) and the output
// projection wo = RowParallelLinear(128 * 128, dim)), and "Attention weights"
// page, excerpt mla-output (the head outputs, flattened, go through wo).
//
// At decode sizes the weight dominates the bytes (wo at dim 7168 is 235 MB
// against 2 MB of tokens), so the kernel is a weight stream on the tensor
// cores.  In the transposed ("swap-AB") form each CTA owns 128 weight rows,
// which sit on the MMA rows, and up to 256 tokens, on the MMA columns:
//     Y^T[n0 .. n0+127][m0 .. m0+NT-1] = W[n0 .., k] . X[m0 .., k]^T
// with the accumulator in TMEM.  TMA brings 64-wide K slices of both operands
// (128-byte swizzle) through a 4-stage ring; one thread issues the MMAs.
// When N / 128 tiles cannot fill the GPU, K is split across CTAs and a second
// kernel sums the per-split partials in split order (no atomics, so the
// result does not depend on scheduling).
#include "common.cuh"
#include "kernels.cuh"
#include "tc05.cuh"

namespace mla {
namespace lin {

using namespace tc;

constexpr int BN = 128;          // weight rows per CTA (MMA M)
constexpr int BK = 64;           // K per stage: one 128-byte swizzle row
constexpr int NT_MAX = 256;      // token columns per CTA (MMA N)
constexpr int STAGES = 4;
constexpr int W_TILE = BN * BK * 2;   // 16 KB
struct Bars {
    uint64_t full[STAGES], empty[STAGES], acc_full, drain;
    uint32_t tmem_base;
};

__host__ __device__ constexpr int stage_bytes(int nt) { return W_TILE + nt * BK * 2; }
__host__ __device__ constexpr int smem_bytes(int nt) { return STAGES * stage_bytes(nt) + 1024; }

__host__ __device__ constexpr uint32_t tmem_cols(int nt) {
    return nt <= 32 ? 32u : nt <= 64 ? 64u : nt <= 128 ? 128u : 256u;
}

// grid: (ceil(N / 128) weight tiles, n_split K ranges, ceil(M / NT) token chunks)
__global__ void __launch_bounds__(128) linear_kernel(const __grid_constant__ CUtensorMap wmap,
                                                     const __grid_constant__ CUtensorMap xmap, int M, int N, int K,
                                                     int NT, int kb_per_split, float *__restrict__ part,
                                                     float *__restrict__ y32, uint16_t *__restrict__ y16,
                                                     int32_t *status, uint64_t wait_ns) {
    extern __shared__ uint8_t smem_raw[];
    __shared__ Bars bars;
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int n0 = blockIdx.x * BN, split = blockIdx.y, m0 = blockIdx.z * NT;
    const int KB = (K + BK - 1) / BK;
    const int kb0 = split * kb_per_split, kb1 = min(KB, kb0 + kb_per_split);
    const int nkb = kb1 - kb0;   // >= 1: the host sizes the splits so that none is empty
    const int SB = stage_bytes(NT);
    const uint32_t ncols = tmem_cols(NT);

    if (tid == 0) {
        for (int s = 0; s < STAGES; ++s) mbar_init(&bars.full[s], 1), mbar_init(&bars.empty[s], 1);
        mbar_init(&bars.acc_full, 1);
        mbar_init(&bars.drain, 1);
        fence_mbar_init();
    }
    if (warp == 2) {
        tmem_alloc(&bars.tmem_base, ncols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = bars.tmem_base;
    const Deadline deadline = make_deadline(wait_ns);
    // X may be the output of the preceding grid of the stream
    grid_dep_wait();

    if (tid == 0) {
        // ---------------------------------------------------------------- TMA producer
        int issued = 0;
        for (int i = 0; i < nkb; ++i) {
            const int s = i % STAGES;
            if (i >= STAGES && !wait_until(&bars.empty[s], ((i / STAGES) - 1) & 1, deadline)) {
                report(status, MLA_DEV_TIMEOUT);
                break;
            }
            uint8_t *st = smem + s * SB;
            mbar_expect_tx(&bars.full[s], SB);
            tma_load_2d(smem_u32(st), &wmap, (kb0 + i) * BK, n0, &bars.full[s]);
            tma_load_2d(smem_u32(st + W_TILE), &xmap, (kb0 + i) * BK, m0, &bars.full[s]);
            issued = i + 1;
        }
        // drain: the loads of the last STAGES issued slices have landed (the
        // earlier ones were consumed before their stage was reissued)
        const uint64_t drain = globaltimer_ns() + DRAIN_NS;
        for (int i = issued > STAGES ? issued - STAGES : 0; i < issued; ++i)
            if (!wait_until(&bars.full[i % STAGES], (i / STAGES) & 1, drain)) {
                report(status, MLA_DEV_TIMEOUT);
                break;
            }
    } else if (tid == 32) {
        // ---------------------------------------------------------------- MMA issuer
        const uint32_t idesc = idesc_bf16(BN, NT, false, false);
        bool ok = true;
        for (int i = 0; i < nkb; ++i) {
            const int s = i % STAGES;
            if (!wait_until(&bars.full[s], (i / STAGES) & 1, deadline)) {
                report(status, MLA_DEV_TIMEOUT);
                ok = false;
                break;
            }
            tc_fence_after();
            const uint32_t sa = smem_u32(smem + s * SB), sb = sa + W_TILE;
#pragma unroll
            for (int kk = 0; kk < BK / 16; ++kk)
                mma_ss(tmem, smem_desc(sa + kk * 32, 16, 1024, 2), smem_desc(sb + kk * 32, 16, 1024, 2), idesc,
                       (i > 0 || kk > 0) ? 1u : 0u);
            mma_commit(&bars.empty[s]);
        }
        if (ok) mma_commit(&bars.acc_full);
        // drain: every MMA issued above has completed before TMEM can be released
        mma_commit(&bars.drain);
        if (!wait_until(&bars.drain, 0, globaltimer_ns() + DRAIN_NS)) report(status, MLA_DEV_TIMEOUT);
    }
    __syncwarp();

    // -------------------------------------------------------------------- epilogue
    // lane = weight row n0 + 32*warp + lane, column j = token m0 + j
    const bool ready = __all_sync(0xffffffffu, wait_until(&bars.acc_full, 0, deadline));
    if (lane == 0 && !ready) report(status, MLA_DEV_TIMEOUT);   // this warp's rows are not written
    if (ready) {
        tc_fence_after();
        // let the next grid of the stream (the split reduction) start its prologue
        if (tid == 0) grid_dep_launch();
        const int n = n0 + 32 * warp + lane;
        const uint32_t trow = tmem + (uint32_t(32 * warp) << 16);
        for (int j0 = 0; j0 < NT; j0 += 16) {
            uint32_t v[16];
            tmem_ld16(trow + j0, v);
            tmem_ld_wait();
            if (n < N) {
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    const int m = m0 + j0 + i;
                    if (m >= M) break;
                    const float f = __uint_as_float(v[i]);
                    if (part)
                        part[((size_t)split * M + m) * N + n] = f;
                    else if (y16)
                        y16[(size_t)m * N + n] = f2bf(f);
                    else
                        y32[(size_t)m * N + n] = f;
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 2) {
        tc_fence_after();
        tmem_dealloc(tmem, ncols);
    }
}

// Y[m][n] = sum over splits, in split order.
__global__ void __launch_bounds__(256) split_reduce_kernel(const float *__restrict__ part, int n_split, long long MN,
                                                           float *__restrict__ y32, uint16_t *__restrict__ y16) {
    grid_dep_wait();
    for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < MN;
         i += (long long)gridDim.x * blockDim.x) {
        float acc = 0.f;
        for (int s = 0; s < n_split; ++s) acc += part[s * MN + i];
        if (y16)
            y16[i] = f2bf(acc);
        else
            y32[i] = acc;
    }
}

}  // namespace lin

size_t linear_workspace(int M, int N, int K, int sms, int *n_split_out, int *kb_per_out) {
    const int tiles = (N + lin::BN - 1) / lin::BN;
    const int chunks = (M + lin::NT_MAX - 1) / lin::NT_MAX;
    const int KB = (K + lin::BK - 1) / lin::BK;
    // split K until the CTAs cover every SM twice (two CTAs fit on an SM at
    // small token counts), keeping at least 4 K slices per split
    int s = (2 * sms) / (tiles * chunks);
    if (s > KB / 4) s = KB / 4;
    if (s < 1) s = 1;
    const int kb_per = (KB + s - 1) / s;
    s = (KB + kb_per - 1) / kb_per;   // no empty split
    if (n_split_out) *n_split_out = s;
    if (kb_per_out) *kb_per_out = kb_per;
    return s > 1 ? (size_t)s * M * N * sizeof(float) : 0;
}

}  // namespace mla

using namespace mla;

static int sm_count() {
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return -1;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return -1;
    return sms;
}

extern "C" size_t mla_linear_workspace_size(int M, int N, int K) {
    if (M < 1 || N < 1 || K < 8 || K % 8 != 0) return 0;
    const int sms = sm_count();
    if (sms <= 0) return 0;
    const size_t ws = linear_workspace(M, N, K, sms, nullptr, nullptr);
    return ws ? ws : 256;   // never 0 for valid sizes (0 means invalid)
}

extern "C" int mla_linear_bf16(const mla_bf16 *x, const mla_bf16 *w, int M, int N, int K, float *y_f32,
                               mla_bf16 *y_bf16, void *workspace, size_t ws_bytes, int32_t *dev_status,
                               mla_stream_t stream) {
    if (!x || !w || (!y_f32 == !y_bf16)) return MLA_ERR_NULL;
    if (!aligned16(x) || !aligned16(w) || (y_f32 && !aligned16(y_f32)) || (y_bf16 && !aligned16(y_bf16)))
        return MLA_ERR_ALIGN;
    if (M < 1 || N < 1 || K < 8 || K % 8 != 0 || (long long)M * N >= (1ll << 40)) return MLA_ERR_SIZE;
    const int sms = sm_count();
    if (sms <= 0) return MLA_ERR_CUDA;
    int n_split = 1, kb_per = 1;
    const size_t need = linear_workspace(M, N, K, sms, &n_split, &kb_per);
    if (need && (!workspace || ws_bytes < need)) return MLA_ERR_WORKSPACE;
    if (need && (reinterpret_cast<uintptr_t>(workspace) & 15u)) return MLA_ERR_ALIGN;
    const int NT = M >= lin::NT_MAX ? lin::NT_MAX : (M + 15) / 16 * 16;
    CUtensorMap wmap, xmap;
    {
        const uint64_t dims[2] = {(uint64_t)K, (uint64_t)N};
        const uint64_t strides[1] = {(uint64_t)K * 2};
        const uint32_t box[2] = {lin::BK, lin::BN};
        if (!make_tmap_bf16(&wmap, w, 2, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B)) return MLA_ERR_CUDA;
    }
    {
        const uint64_t dims[2] = {(uint64_t)K, (uint64_t)M};
        const uint64_t strides[1] = {(uint64_t)K * 2};
        const uint32_t box[2] = {lin::BK, (uint32_t)NT};
        if (!make_tmap_bf16(&xmap, x, 2, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B)) return MLA_ERR_CUDA;
    }
    const int smem = lin::smem_bytes(NT);
    static std::atomic<bool> smem_set[64];
    if (!smem_attr_once(smem_set, lin::linear_kernel, lin::smem_bytes(lin::NT_MAX))) return MLA_ERR_CUDA;
    cudaStream_t s = (cudaStream_t)stream;
    const dim3 grid((N + lin::BN - 1) / lin::BN, n_split, (M + NT - 1) / NT);
    float *part = n_split > 1 ? static_cast<float *>(workspace) : nullptr;
    if (launch_k(true, lin::linear_kernel, grid, dim3(128), smem, s, wmap, xmap, M, N, K, NT, kb_per, part, y_f32,
                 reinterpret_cast<uint16_t *>(y_bf16), dev_status, wait_limit_ns()) != cudaSuccess)
        return MLA_ERR_CUDA;
    int launches = 1;
    if (n_split > 1) {
        const long long MN = (long long)M * N;
        const long long want = (MN + 255) / 256;
        const int blocks = int(want < (long long)sms * 8 ? want : (long long)sms * 8);
        if (launch_k(true, lin::split_reduce_kernel, dim3(blocks), dim3(256), 0, s, (const float *)part, n_split,
                     MN, y_f32, reinterpret_cast<uint16_t *>(y_bf16)) != cudaSuccess)
            return MLA_ERR_CUDA;
        ++launches;
    }
    count_launches(launches);
    return MLA_OK;
}
