/*
 * mla_decode.h -- C ABI of the B300 (sm_103a) library for one decode step of
 * absorbed, top-k-sparse latent attention (DeepSeek-V3.2-Exp sparse MLA).
 *
 * The step, as the DeepSeek-V3.2-Exp atlas pages state it ("Rotated query
 * part" / "Query content heads" / "Attention weights", excerpt mla-decode):
 *
 *   q~[b,h,:]   = q_nope[b,h,:] . W_UK[h]                     (key absorption)
 *   s[b,h,t]    = (q~[b,h,:] . kv[b,t,:] + rope(q_pe)[b,h,:] . pe[b,t,:]) * scale
 *   s[b,h,t]   += 0 for t in topk_idx[b,:], -inf otherwise     (selection mask)
 *   p           = softmax_t(s)
 *   o[b,h,:]    = sum_t p[b,h,t] kv[b,t,:]
 *   out[b,h,:]  = W_UV[h] . o[b,h,:]                          (value up-projection)
 *
 * with wkv_b [128*256, 512] viewed [128, 256, 512]: rows 0..127 of head h are
 * W_UK[h] (128 x 512), rows 128..255 are W_UV[h] (128 x 512).
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - H = 128 heads, d_nope = 128, d_rope = 64, d_v = 128, kv_lora = 512 are
 *    fixed (the kernels are specialised for them).
 *  - mla_bf16 is the raw bit pattern of an IEEE bfloat16.
 *  - Every tensor pointer is a DEVICE pointer (cudaMalloc / torch CUDA memory)
 *    unless stated otherwise, row-major and contiguous, 16-byte aligned.
 *  - The caller owns every buffer (inputs, outputs, workspace, status word).
 *    The library allocates nothing and keeps no state between calls, except
 *    cached per-device properties read on first use.
 *  - Calls are asynchronous on `stream` (a cudaStream_t; NULL = legacy default
 *    stream).  A call returns after enqueueing its kernels.
 *  - Return value: MLA_OK (0) on success; a negative MLA_ERR_* code when an
 *    argument check fails on the host (nothing is enqueued then), or
 *    MLA_ERR_CUDA when a launch fails.  No exception crosses the ABI.
 *  - Kernels are chained on the stream by programmatic dependent launch.
 *    The attention kernel starts gathering kv_cache / pe_cache rows (per
 *    topk_idx and end_pos) while the grid before it may still be running; it
 *    waits for that grid before reading q_lat or writing any output.  These
 *    four inputs must therefore be complete before the call is enqueued (any
 *    ordinary kernel, copy or event before it guarantees that); only a kernel
 *    that itself triggers dependent launch early could break this.
 *  - Conditions only the device can see (an end_pos outside [1, S_cap], a
 *    position outside the rotary table, a bounded wait that ran out) are OR-ed
 *    as MLA_DEV_* bits into *dev_status (when dev_status is non-NULL); read it
 *    after synchronising the stream.  Affected sequences produce zeros.  A
 *    repeated position in a selection row is not detected on the decode path;
 *    mla_check_selection finds it on request.
 */
#ifndef MLA_DECODE_H
#define MLA_DECODE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef uint16_t mla_bf16;
typedef struct CUstream_st *mla_stream_t; /* same type as cudaStream_t */

#define MLA_N_HEADS 128
#define MLA_D_NOPE 128
#define MLA_D_ROPE 64
#define MLA_D_V 128
#define MLA_KV_LORA 512
#define MLA_Q_LAT 576 /* kv_lora + d_rope */

/* host-side return codes */
#define MLA_OK 0
#define MLA_ERR_NULL (-1)        /* a required pointer is NULL */
#define MLA_ERR_ALIGN (-2)       /* a pointer is not 16-byte aligned */
#define MLA_ERR_SIZE (-3)        /* a size argument is out of range */
#define MLA_ERR_WORKSPACE (-4)   /* workspace smaller than required */
#define MLA_ERR_CUDA (-5)        /* a CUDA launch or query failed */
#define MLA_ERR_DEVICE (-6)      /* current device is not sm_103 */

/* device-side status bits (OR-ed into *dev_status) */
#define MLA_DEV_BAD_END_POS 1    /* end_pos[b] < 1 or > S_cap: sequence b skipped */
#define MLA_DEV_BAD_POSITION 2   /* end_pos[b]-1 outside the rotary table */
#define MLA_DEV_TIMEOUT 4        /* a bounded on-chip wait gave up */
#define MLA_DEV_SCORE_RANGE 8    /* a partial score exceeded 2048 in magnitude: the
                                    exchanged fp16 copy may be off by a whole unit
                                    (see mla_sparse_decode, precision) */
#define MLA_DEV_DUPLICATE_INDEX 16 /* a selection row repeats a valid position
                                      (set by mla_check_selection only) */

/* Rotary / YaRN parameters.  Defaults (mla_rope_params_default) are those of
 * the "Transformer blocks" page, excerpt model-args: max_seq_len 16384,
 * original_seq_len 4096, rope_theta 1e4, rope_factor 40, beta_fast 32,
 * beta_slow 1, mscale 1, rope_dim 64. */
typedef struct mla_rope_params {
    int32_t rope_dim;         /* must be 64 */
    int32_t max_seq_len;      /* rows of the rotary table */
    int32_t original_seq_len; /* YaRN is applied when max_seq_len > this */
    int32_t reserved;         /* set to 0 */
    double rope_theta;
    double rope_factor;
    double beta_fast;
    double beta_slow;
    double mscale;
} mla_rope_params;

/* Fill *p with the defaults above (host only). */
void mla_rope_params_default(mla_rope_params *p);

/* Softmax scale of the step ("Query heads" page, excerpt mla-init):
 * qk_head_dim^-0.5, times (0.1*mscale*ln(rope_factor) + 1)^2 when
 * max_seq_len > original_seq_len.  Host-only helper; qk_head_dim = 192 for
 * this block.  Returns a negative value when p is NULL or qk_head_dim <= 0. */
double mla_softmax_scale(const mla_rope_params *p, int qk_head_dim);

/* rope_freqs_init -- the rotary coefficient table ("Transformer blocks" page,
 * RoPE coefficients panel, excerpt rope).
 *   cis  [max_seq_len][32][2] fp32, device, written: (cos, sin) of t * f'_i,
 *        f'_i = YaRN-blended 1 / theta^(2i/64).  Angles and sincos are
 *        evaluated in fp64 on the device and stored rounded to fp32.
 *   p    host pointer to the parameters (copied by value at the call).
 * Errors: MLA_ERR_NULL, MLA_ERR_ALIGN, MLA_ERR_SIZE (rope_dim != 64,
 * max_seq_len < 1 or > 1<<24, theta/factor <= 0, beta_fast <= 0 or
 * beta_slow <= 0). */
int rope_freqs_init(float *cis, const mla_rope_params *p, mla_stream_t stream);

/* mla_rope_apply -- interleaved rotary embedding of the query's rotary part
 * ("Rotated query part" page, excerpt apply-rope): each pair
 * (x[2i], x[2i+1]) is multiplied, as a complex number, by cis[pos_b][i] in
 * fp32, with pos_b = end_pos[b] - 1.
 *   q_pe      [B][128][64] bf16, device
 *   cis       [max_seq_len][32][2] fp32 from rope_freqs_init
 *   end_pos   [B] int32, device
 *   q_pe_rot  [B][128][64] fp32, device, written (zeros for a sequence whose
 *             position is outside [0, max_seq_len): MLA_DEV_BAD_POSITION)
 * Errors: MLA_ERR_NULL, MLA_ERR_ALIGN, MLA_ERR_SIZE (B < 1 or > 65535,
 * max_seq_len < 1). */
int mla_rope_apply(const mla_bf16 *q_pe, const float *cis, int max_seq_len, const int32_t *end_pos,
                   int B, float *q_pe_rot, int32_t *dev_status, mla_stream_t stream);

/* mla_rope_apply_layout -- rotary embedding of 64-wide rotary vectors with a
 * selectable pair layout ("Rotated query part" page, excerpt apply-rope, its
 * `interleaved` argument), at position end_pos[b] - 1, in fp32:
 *   interleaved = 1: pair i is (x[2i], x[2i+1]), rotated in place (the query
 *                    layout; the same result as mla_rope_apply);
 *   interleaved = 0: pair i is (x[i], x[i+32]); the real parts are written to
 *                    features 0..31 and the imaginary parts to 32..63 (the
 *                    layout the page's indexer uses).
 *   x   [B][n_heads][64] bf16, device; out [B][n_heads][64] fp32, device, written
 *       (zeros for a sequence whose position is outside the table:
 *       MLA_DEV_BAD_POSITION).
 * Errors: MLA_ERR_NULL, MLA_ERR_ALIGN, MLA_ERR_SIZE (B < 1 or > 65535,
 * n_heads < 1 or > 1024, max_seq_len < 1, interleaved not 0 or 1). */
int mla_rope_apply_layout(const mla_bf16 *x, const float *cis, int max_seq_len, const int32_t *end_pos, int B,
                          int n_heads, int interleaved, float *out, int32_t *dev_status, mla_stream_t stream);

/* mla_absorb_q -- the query of the latent attention: key absorption
 * ("Query content heads" page, excerpt mla-decode, first einsum) with the
 * RoPE of q_pe fused in:
 *   q_lat[b,h,0:512]   = bf16( sum_d q_nope[b,h,d] * W_UK[h][d][:] )  (fp32 accumulate)
 *   q_lat[b,h,512:576] = bf16( rope(q_pe[b,h,:], pos_b) )
 *   q_nope [B][128][128] bf16, q_pe [B][128][64] bf16, cis as above,
 *   end_pos [B] int32, wkv_b [32768][512] bf16, q_lat [B][128][576] bf16 (written).
 * Errors: MLA_ERR_NULL, MLA_ERR_ALIGN, MLA_ERR_SIZE (B < 1 or > 4096). */
int mla_absorb_q(const mla_bf16 *q_nope, const mla_bf16 *q_pe, const float *cis, int max_seq_len,
                 const int32_t *end_pos, const mla_bf16 *wkv_b, int B, mla_bf16 *q_lat,
                 int32_t *dev_status, mla_stream_t stream);

/* mla_absorb_q_tokens -- mla_absorb_q for T query tokens per sequence
 * (multi-token decode).  Row r = b*T + s is token s of sequence b; its
 * rotary part is rotated at position end_pos[b] - T + s.
 *   q_nope [n_seq][T][128][128], q_pe [n_seq][T][128][64] bf16,
 *   end_pos [n_seq] int32 (cached tokens AFTER the T new ones),
 *   q_lat [n_seq][T][128][576] bf16 (written).  T = 1 is mla_absorb_q.
 * Errors: as mla_absorb_q, with MLA_ERR_SIZE for n_seq or T < 1 or
 * n_seq*T > 4096. */
int mla_absorb_q_tokens(const mla_bf16 *q_nope, const mla_bf16 *q_pe, const float *cis, int max_seq_len,
                        const int32_t *end_pos, const mla_bf16 *wkv_b, int n_seq, int T, mla_bf16 *q_lat,
                        int32_t *dev_status, mla_stream_t stream);

/* Bytes of device workspace mla_sparse_decode needs for B query rows (B
 * sequences, or n_seq*T rows for mla_sparse_decode_tokens) whose selection
 * rows hold K entries.  0 when B or K is out of range. */
size_t mla_sparse_decode_workspace_size(int B, int K);

/* mla_sparse_decode -- scores of every head against the selected rows of the
 * shared 576-wide cache, softmax over the selected set, probability-weighted
 * sum of the latent rows, and (when wkv_b is given) the value up-projection
 * ("Attention weights" page, excerpt mla-decode, scores .. last einsum).
 *   q_lat     [B][128][576] bf16 (from mla_absorb_q)
 *   kv_cache  [B][S_cap][512] bf16, pe_cache [B][S_cap][64] bf16
 *   topk_idx  [B][K] int32: positions selected for sequence b.  Entries < 0
 *             or >= end_pos[b] are padding and ignored.  Valid entries of a
 *             row must be distinct (the selection is a set; a repeated
 *             position would be counted twice).
 *   end_pos   [B] int32: cached keys of sequence b (1 <= end_pos <= S_cap)
 *   softmax_scale: multiplies the raw scores (see mla_softmax_scale)
 *   wkv_b     NULL, or [32768][512] bf16 for the fused up-projection
 *   out       wkv_b != NULL: [B][128][128] fp32 head outputs;
 *             wkv_b == NULL: [B][128][512] fp32 normalised latent outputs o.
 *             A sequence with no valid selected position yields zeros.
 *   workspace device scratch of at least mla_sparse_decode_workspace_size(B, K)
 *             bytes, 256-byte aligned; contents on entry do not matter.
 *   dev_status optional device int32, MLA_DEV_* bits OR-ed in.
 * Precision: bf16 operands, fp32 accumulation, fp32 softmax.  The 576-wide
 * score dot product is split in two halves computed on two SMs; each half's
 * raw (unscaled) partial score reaches the other SM rounded to fp16, i.e. to
 * 11 significant bits, so a score carries an extra error of at most
 * 2^-12 * |partial|.  The seeded workloads reach |partial| of about 50 and
 * the GPU tests check partials up to about 800 (logits softmax_scale *
 * |partial| up to about 110) against the tolerance; a partial beyond 2048
 * sets MLA_DEV_SCORE_RANGE, since the error of one exchanged copy can then
 * reach a whole unit of the raw score.  With wkv_b, o is rounded to bf16 as
 * the up-projection's operand; when the selection of one or two query rows
 * is split over several SM pairs, each split's normalised o is kept as bf16,
 * and the up-projection merges the splits and multiplies in fp32.
 * Errors: MLA_ERR_NULL, MLA_ERR_ALIGN, MLA_ERR_SIZE (B < 1 or > 4096,
 * K < 1 or > 1<<20, S_cap < 1), MLA_ERR_WORKSPACE. */
int mla_sparse_decode(const mla_bf16 *q_lat, const mla_bf16 *kv_cache, const mla_bf16 *pe_cache,
                      int S_cap, const int32_t *topk_idx, int K, const int32_t *end_pos, int B,
                      float softmax_scale, const mla_bf16 *wkv_b, float *out, void *workspace,
                      size_t ws_bytes, int32_t *dev_status, mla_stream_t stream);

/* mla_sparse_decode_tokens -- mla_sparse_decode for T query tokens per
 * sequence (multi-token decode; the "Attention weights" page notes that the
 * causal mask is merged into the selection).  Row r = b*T + s is token s of
 * sequence b, at position pos = end_pos[b] - T + s; it attends to the
 * positions of its own selection row topk_idx[r] that are <= pos (the
 * selection merged with the causal mask; entries > pos count as padding).
 *   q_lat    [n_seq][T][128][576] bf16 (mla_absorb_q_tokens)
 *   kv_cache [n_seq][S_cap][512], pe_cache [n_seq][S_cap][64] bf16 (the T new
 *            rows already appended, e.g. by mla_cache_append)
 *   topk_idx [n_seq][T][K] int32, end_pos [n_seq] int32 (T <= end_pos <= S_cap,
 *            else MLA_DEV_BAD_END_POS and zeros for that sequence)
 *   out      [n_seq][T][128][128] (wkv_b given) or [n_seq][T][128][512]:
 *            fp32 when out_bf16 = 0, bf16 (rounded once from the fp32
 *            result) when out_bf16 = 1 -- the form mla_linear_bf16 takes as
 *            the input of the output projection wo.
 *   workspace at least mla_sparse_decode_workspace_size(n_seq*T, K) bytes.
 * T = 1 with out_bf16 = 0 is mla_sparse_decode.  Errors: as
 * mla_sparse_decode, with MLA_ERR_SIZE for n_seq or T < 1, n_seq*T > 4096 or
 * out_bf16 not 0 or 1. */
int mla_sparse_decode_tokens(const mla_bf16 *q_lat, const mla_bf16 *kv_cache, const mla_bf16 *pe_cache, int S_cap,
                             const int32_t *topk_idx, int K, const int32_t *end_pos, int n_seq, int T,
                             float softmax_scale, const mla_bf16 *wkv_b, void *out, int out_bf16, void *workspace,
                             size_t ws_bytes, int32_t *dev_status, mla_stream_t stream);

/* mla_out_up -- value up-projection alone ("Attention weights" page, excerpt
 * mla-decode, last einsum): out[b,h,d] = sum_c o_lat[b,h,c] * W_UV[h][d][c],
 * with o_lat rounded to bf16 and fp32 accumulation.
 *   o_lat [B][128][512] fp32, wkv_b [32768][512] bf16, out [B][128][128] fp32.
 * Errors: MLA_ERR_NULL, MLA_ERR_ALIGN, MLA_ERR_SIZE (B < 1 or > 4096). */
int mla_out_up(const float *o_lat, const mla_bf16 *wkv_b, int B, float *out, mla_stream_t stream);

/* mla_check_selection -- validation of the selection rows, for callers that
 * want to verify the distinct-positions precondition of mla_sparse_decode
 * (a debugging aid: no other entry point calls it, and it is not needed for
 * correct input).  The selection is a set ("Attention weights" page, excerpt
 * mla-decode: zeros scattered into a row of -inf), while the attention
 * kernels add one term per valid entry, so a position repeated among a row's
 * valid entries would be counted twice.
 *   topk_idx   [n_seq][T][K] int32, as for mla_sparse_decode_tokens (T = 1:
 *              mla_sparse_decode's [B][K])
 *   end_pos    [n_seq] int32
 *   dev_status device int32 (required): MLA_DEV_DUPLICATE_INDEX is OR-ed in
 *              when some row r = b*T + s holds a position t twice with
 *              0 <= t <= end_pos[b] - T + s (the positions the row sees);
 *              padding (entries < 0 or beyond that) is never flagged,
 *              repeated or not.  A sequence whose end_pos is < T or > S_cap
 *              is skipped and flagged MLA_DEV_BAD_END_POS, as the decode
 *              would skip it.
 * One kernel, one block per row, a bitmap of S_cap bits in shared memory.
 * Errors: MLA_ERR_NULL, MLA_ERR_ALIGN, MLA_ERR_SIZE (n_seq or T < 1,
 * n_seq*T > 4096, K < 1 or > 1<<20, S_cap < 1 or > MLA_CHECK_MAX_S_CAP). */
#define MLA_CHECK_MAX_S_CAP (1 << 20)
int mla_check_selection(const int32_t *topk_idx, int K, const int32_t *end_pos, int n_seq, int T, int S_cap,
                        int32_t *dev_status, mla_stream_t stream);

/* mla_cache_append -- write T new tokens per sequence into the caches ("Query
 * heads" page, excerpt mla-init: the joint down-projection wkv_a emits the
 * 512 latent features and the 64-wide shared rotary key; kv_norm is an
 * RMSNorm over the latent; "Attention weights" page, excerpt mla-decode:
 * kv_cache / pe_cache are read up to end_pos).  The pages do not print the
 * write; the plain reading is: token s of sequence b sits at position
 * pos = end_pos[b] - T + s, and
 *   kv_cache[b][pos][:] = bf16( x * w / sqrt(mean(x^2) + eps) ),  x = kv_a[b][s][0:512]
 *   pe_cache[b][pos][:] = bf16( rope_interleaved(kv_a[b][s][512:576], pos) )
 * with fp32 arithmetic (the rotation as in mla_rope_apply).
 *   kv_a      [B][T][576] bf16, device: the wkv_a output of the new tokens.
 *   kv_norm_w [512] fp32, device (a bf16 weight widens exactly).
 *   eps       RMSNorm epsilon (>= 0; 1e-6 in DeepSeek-V3 checkpoints).
 *   cis       rotary table [max_seq_len][32][2] fp32 (rope_freqs_init).
 *   end_pos   [B] int32: cached tokens of sequence b AFTER the append.
 *   kv_cache  [B][S_cap][512] bf16, pe_cache [B][S_cap][64] bf16, device:
 *             rows end_pos[b]-T .. end_pos[b]-1 are written, nothing else.
 * A sequence with end_pos[b] < T or > S_cap is skipped (MLA_DEV_BAD_END_POS);
 * a token whose position is outside the rotary table is skipped
 * (MLA_DEV_BAD_POSITION).
 * Errors: MLA_ERR_NULL, MLA_ERR_ALIGN, MLA_ERR_SIZE (B, T, S_cap or
 * max_seq_len < 1, B*T >= 2^31, eps negative or NaN). */
int mla_cache_append(const mla_bf16 *kv_a, const float *kv_norm_w, float eps, const float *cis, int max_seq_len,
                     const int32_t *end_pos, int B, int T, mla_bf16 *kv_cache, mla_bf16 *pe_cache, int S_cap,
                     int32_t *dev_status, mla_stream_t stream);

/* mla_linear_bf16 -- token-by-weight projection Y = X . W^T, the layout of
 * the pages' Linear layers on either side of the attention ("Query heads"
 * page, excerpt mla-init: wkv_a = Linear(dim, 576) makes the kv_a rows that
 * mla_cache_append takes; wo = RowParallelLinear(128*128, dim); "Attention
 * weights" page, excerpt mla-output: wo applied to the flattened head
 * outputs).  bf16 operands, fp32 accumulation on the tensor cores:
 *   Y[m][n] = sum_k X[m][k] * W[n][k]
 *   x  [M][K] bf16, w [N][K] bf16 (device, 16-byte aligned, K % 8 == 0).
 *   Exactly one of y_f32 [M][N] fp32 / y_bf16 [M][N] bf16 is non-NULL.
 *   workspace: mla_linear_workspace_size(M, N, K) bytes of device scratch
 *   (16-byte aligned; NULL allowed when that size is 256, i.e. no split of K
 *   is needed on the current device).  When K is split across CTAs the
 *   partial sums are added in a fixed order, so results are reproducible.
 * Errors: MLA_ERR_NULL (x or w NULL, or not exactly one output),
 * MLA_ERR_ALIGN, MLA_ERR_SIZE (M, N < 1, K < 8 or K % 8 != 0),
 * MLA_ERR_WORKSPACE, MLA_ERR_CUDA. */
size_t mla_linear_workspace_size(int M, int N, int K);
int mla_linear_bf16(const mla_bf16 *x, const mla_bf16 *w, int M, int N, int K, float *y_f32, mla_bf16 *y_bf16,
                    void *workspace, size_t ws_bytes, int32_t *dev_status, mla_stream_t stream);

/* mla_weight_dequant_fp8 -- block-scaled fp8 weight to bf16 (the pages'
 * weight_dequant(wkv_b.weight, wkv_b.scale), "Rotated query part" page,
 * excerpt mla-decode, run once and kept as the wkv_b of the absorbed path):
 *   out[r][c] = bf16_rn( fp32( e4m3(w[r][c]) * scale[r / block][c / block] ) )
 * The pages name the call but not its format; this entry reads it as OCP
 * FP8 E4M3 codes (bias 7, no infinities, S.1111.111 = NaN) with one fp32
 * multiplier per block x block tile (block 128 for DeepSeek-V3 checkpoints).
 *   w     [rows][cols] uint8 e4m3 codes, device.
 *   scale [ceil(rows/block)][ceil(cols/block)] fp32, device, 4-byte aligned.
 *   out   [rows][cols] bf16, device, 2-byte aligned, written.  A NaN code
 *         gives a NaN.
 * Any rows, cols and block >= 1; when cols and block are multiples of 16 and
 * w and out are 16-byte aligned the kernel moves 16 elements per access.
 * For wkv_b: rows 32768, cols 512, block 128, scale [256][4].
 * Errors: MLA_ERR_NULL, MLA_ERR_ALIGN, MLA_ERR_SIZE (rows, cols or block < 1,
 * rows*cols > 2^40), MLA_ERR_CUDA. */
int mla_weight_dequant_fp8(const uint8_t *w, const float *scale, int rows, int cols, int block, mla_bf16 *out,
                           mla_stream_t stream);

/* mla_sparse_decode_static_ws -- mla_sparse_decode without a caller-supplied
 * workspace.  The pages have no counterpart to this call; it exists for
 * callers that cannot allocate device memory (a plugin host that owns every
 * buffer, a serving loop where an allocator call could stall the device, a
 * fixed memory plan).  They pass inputs and outputs as for mla_sparse_decode;
 * the scratch comes from one array of MLA_STATIC_WS_BYTES compiled into the
 * library's device image (each GPU that loads the library reserves it until
 * the process exits).  The call allocates nothing.
 *   - Arguments, layouts and results are those of mla_sparse_decode.
 *   - Returns MLA_ERR_SIZE when mla_sparse_decode_workspace_size(B, K) is 0
 *     or exceeds MLA_STATIC_WS_BYTES (the bf16 latent output alone takes
 *     B*128*512*2 bytes, so B <= 256).
 *   - The first call on a device looks up the array's device address with
 *     that device current; make that first call before any stream capture.
 *     The address is remembered with the context it belongs to: after a
 *     cudaDeviceReset (a new primary context) the next call looks it up
 *     again, so that call too should come before any capture.
 *   - Every call on a device shares the one array and leaves its contents
 *     behind; nothing in it needs to start at zero.  Calls whose kernels
 *     overlap on the GPU (other streams, other host threads) race on it:
 *     order them on one stream. */
#define MLA_STATIC_WS_BYTES (32u << 20)
int mla_sparse_decode_static_ws(const mla_bf16 *q_lat, const mla_bf16 *kv_cache, const mla_bf16 *pe_cache,
                                int S_cap, const int32_t *topk_idx, int K, const int32_t *end_pos, int B,
                                float softmax_scale, const mla_bf16 *wkv_b, float *out, int32_t *dev_status,
                                mla_stream_t stream);

/* Profiling hook for the calling host thread (the library's only mutable
 * state, and it is per thread).  While set:
 *   - every entry point adds the number of kernels it enqueues to
 *     *launch_count (when launch_count is non-NULL);
 *   - mla_sparse_decode records ev_start (a cudaEvent_t) on its stream just
 *     before its attention kernel and ev_stop just after it (when both are
 *     non-NULL), so the attention kernel alone can be timed.
 * Pass NULL for all three to clear.  Returns MLA_OK. */
int mla_profile_hook(void *ev_start, void *ev_stop, int64_t *launch_count);

/* Limit, in nanoseconds, of every bounded on-chip wait of the kernels
 * (default 2e9, i.e. 2 s; 0 is taken as 1).  The pages have no counterpart:
 * it is the failure-detection knob of this library.  A kernel whose wait runs
 * out sets MLA_DEV_TIMEOUT in *dev_status, then waits (for at most 1 s more)
 * for the copies and MMAs it has already issued, releases its tensor memory
 * and returns, so the context stays usable.  Process-wide; read when a kernel
 * is launched (a CUDA graph keeps the value captured with it).  Meant for
 * tests that drive a wait past its limit; returns the previous limit. */
uint64_t mla_set_wait_limit_ns(uint64_t ns);

/* Static description of a return code or of a set of MLA_DEV_* bits
 * (pass the negative return code, or the status word as a positive value). */
const char *mla_status_string(int code);

#ifdef __cplusplus
}
#endif

#endif /* MLA_DECODE_H */
