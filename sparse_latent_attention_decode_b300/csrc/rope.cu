// Rotary coefficient table and interleaved rotary embedding.
//
// Sources: DeepSeek-V3.2-Exp atlas, "Transformer blocks" page (RoPE
// coefficients panel, excerpts rope and model-args) for the table, and
// "Rotated query part" page (excerpt apply-rope) for the pair rotation.
#include "common.cuh"

namespace mla {

struct RopeArgs {
    int dim, max_seq_len, original_seq_len;
    double theta, factor, beta_fast, beta_slow;
};

// f'_i: 1/theta^(2i/dim), blended with f_i/factor by the YaRN linear ramp
// between the correction dims low = floor(cd(beta_fast)) and
// high = ceil(cd(beta_slow)) (clamped to [0, dim-1]), where
// cd(n) = dim * ln(L0 / (2 pi n)) / (2 ln theta).  All in fp64.
__device__ double yarn_freq(int i, const RopeArgs &a) {
    double f = 1.0 / pow(a.theta, (2.0 * i) / a.dim);
    if (a.max_seq_len > a.original_seq_len) {
        const double two_pi = 6.283185307179586476925286766559;
        const double denom = 2.0 * log(a.theta);
        double lo = floor(a.dim * log(a.original_seq_len / (a.beta_fast * two_pi)) / denom);
        double hi = ceil(a.dim * log(a.original_seq_len / (a.beta_slow * two_pi)) / denom);
        lo = fmax(lo, 0.0);
        hi = fmin(hi, double(a.dim - 1));
        if (lo == hi) hi += 0.001;
        double r = fmin(fmax((i - lo) / (hi - lo), 0.0), 1.0);
        double smooth = 1.0 - r;
        f = f / a.factor * (1.0 - smooth) + f * smooth;
    }
    return f;
}

__global__ void rope_freqs_kernel(float2 *__restrict__ cis, RopeArgs a) {
    const int half = a.dim / 2;
    const long long n = (long long)a.max_seq_len * half;
    for (long long k = blockIdx.x * (long long)blockDim.x + threadIdx.x; k < n;
         k += (long long)gridDim.x * blockDim.x) {
        const int t = int(k / half), i = int(k % half);
        const double ang = double(t) * yarn_freq(i, a);
        double s, c;
        sincos(ang, &s, &c);
        cis[k] = make_float2(float(c), float(s));
    }
}

// One thread per (sequence, head, pair): rotate pair i by cis[end_pos[b]-1][i]
// in fp32.  Interleaved layout: the pair is (x[2i], x[2i+1]) and is written
// back in place; half-split layout (the indexer's): the pair is (x[i], x[i+32])
// and the real / imaginary parts go to slots i and i+32.
__global__ void rope_apply_kernel(const uint16_t *__restrict__ x, const float2 *__restrict__ cis, int max_seq_len,
                                  const int32_t *__restrict__ end_pos, int B, int n_heads, int interleaved,
                                  float *__restrict__ out, int32_t *status) {
    const long long n = (long long)B * n_heads * NPAIR;
    for (long long k = blockIdx.x * (long long)blockDim.x + threadIdx.x; k < n;
         k += (long long)gridDim.x * blockDim.x) {
        const int i = int(k % NPAIR);
        const long long row = k / NPAIR;   // (b, head)
        const int b = int(row / n_heads);
        const int pos = end_pos[b] - 1;
        const uint16_t *xr = x + row * DR;
        float *yr = out + row * DR;
        const int s0 = interleaved ? 2 * i : i, s1 = interleaved ? 2 * i + 1 : i + NPAIR;
        if (pos < 0 || pos >= max_seq_len) {
            yr[s0] = 0.f, yr[s1] = 0.f;
            if (i == 0 && row % n_heads == 0) report(status, MLA_DEV_BAD_POSITION);
            continue;
        }
        const float x0 = bf2f(xr[s0]), x1 = bf2f(xr[s1]);
        const float2 cs = cis[(long long)pos * NPAIR + i];
        yr[s0] = x0 * cs.x - x1 * cs.y;
        yr[s1] = x0 * cs.y + x1 * cs.x;
    }
}

}  // namespace mla

using namespace mla;

extern "C" void mla_rope_params_default(mla_rope_params *p) {
    if (!p) return;
    p->rope_dim = 64;
    p->max_seq_len = 4096 * 4;
    p->original_seq_len = 4096;
    p->reserved = 0;
    p->rope_theta = 10000.0;
    p->rope_factor = 40.0;
    p->beta_fast = 32.0;
    p->beta_slow = 1.0;
    p->mscale = 1.0;
}

extern "C" double mla_softmax_scale(const mla_rope_params *p, int qk_head_dim) {
    if (!p || qk_head_dim <= 0) return -1.0;
    double s = 1.0 / sqrt(double(qk_head_dim));
    if (p->max_seq_len > p->original_seq_len) {
        double m = 0.1 * p->mscale * log(p->rope_factor) + 1.0;
        s *= m * m;
    }
    return s;
}

extern "C" int rope_freqs_init(float *cis, const mla_rope_params *p, mla_stream_t stream) {
    if (!cis || !p) return MLA_ERR_NULL;
    if (!aligned16(cis)) return MLA_ERR_ALIGN;
    if (p->rope_dim != DR || p->max_seq_len < 1 || p->max_seq_len > (1 << 24) || p->original_seq_len < 1 ||
        !(p->rope_theta > 0.0) || !(p->rope_factor > 0.0) || !(p->beta_fast > 0.0) || !(p->beta_slow > 0.0))
        return MLA_ERR_SIZE;
    RopeArgs a{p->rope_dim, p->max_seq_len, p->original_seq_len, p->rope_theta, p->rope_factor,
               p->beta_fast, p->beta_slow};
    const long long n = (long long)p->max_seq_len * NPAIR;
    const int threads = 256;
    const int blocks = int((n + threads - 1) / threads < 148 * 16 ? (n + threads - 1) / threads : 148 * 16);
    rope_freqs_kernel<<<blocks, threads, 0, (cudaStream_t)stream>>>(reinterpret_cast<float2 *>(cis), a);
    count_launches(1);
    return cudaGetLastError() == cudaSuccess ? MLA_OK : MLA_ERR_CUDA;
}

static int rope_apply(const mla_bf16 *x, const float *cis, int max_seq_len, const int32_t *end_pos, int B,
                      int n_heads, int interleaved, float *out, int32_t *dev_status, mla_stream_t stream) {
    if (!x || !cis || !end_pos || !out) return MLA_ERR_NULL;
    if (!aligned16(x) || !aligned16(cis) || !aligned16(out)) return MLA_ERR_ALIGN;
    if (B < 1 || B > 65535 || n_heads < 1 || n_heads > 1024 || max_seq_len < 1 ||
        (interleaved != 0 && interleaved != 1))
        return MLA_ERR_SIZE;
    const long long n = (long long)B * n_heads * NPAIR;
    const int threads = 256;
    const long long want = (n + threads - 1) / threads;
    const int blocks = int(want < 148 * 32 ? want : 148 * 32);
    rope_apply_kernel<<<blocks, threads, 0, (cudaStream_t)stream>>>(x, reinterpret_cast<const float2 *>(cis),
                                                                    max_seq_len, end_pos, B, n_heads, interleaved,
                                                                    out, dev_status);
    count_launches(1);
    return cudaGetLastError() == cudaSuccess ? MLA_OK : MLA_ERR_CUDA;
}

extern "C" int mla_rope_apply(const mla_bf16 *q_pe, const float *cis, int max_seq_len, const int32_t *end_pos,
                              int B, float *q_pe_rot, int32_t *dev_status, mla_stream_t stream) {
    return rope_apply(q_pe, cis, max_seq_len, end_pos, B, H, 1, q_pe_rot, dev_status, stream);
}

extern "C" int mla_rope_apply_layout(const mla_bf16 *x, const float *cis, int max_seq_len, const int32_t *end_pos,
                                     int B, int n_heads, int interleaved, float *out, int32_t *dev_status,
                                     mla_stream_t stream) {
    return rope_apply(x, cis, max_seq_len, end_pos, B, n_heads, interleaved, out, dev_status, stream);
}

namespace mla {
ProfileHook &profile_hook() {
    static thread_local ProfileHook h;
    return h;
}
}  // namespace mla

extern "C" int mla_profile_hook(void *ev_start, void *ev_stop, int64_t *launch_count) {
    ProfileHook &h = profile_hook();
    h.start = static_cast<cudaEvent_t>(ev_start);
    h.stop = static_cast<cudaEvent_t>(ev_stop);
    h.launches = launch_count;
    return MLA_OK;
}
