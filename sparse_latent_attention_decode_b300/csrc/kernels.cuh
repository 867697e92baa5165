// Launchers and host helpers shared between translation units of the library.
#pragma once

#include <cuda.h>

#include <atomic>

#include "common.cuh"

namespace mla {

// Value up-projection of the normalised latent output o, given either as
// fp32 (o_f32, the standalone entry point) or as bf16 (o_b16, written by the
// attention path); exactly one of them is non-NULL.  The head outputs go to
// out (fp32) or, when out_b16 is non-NULL, to out_b16 (bf16).
// With part_o non-NULL (and o_f32, o_b16 NULL) the operand is merged from
// the attention kernel's split partials (part_o as bf16, written so by a
// launch_attn with merge_later; part_lse; n_split per row).
int launch_out_up(const float *o_f32, const uint16_t *o_b16, const uint16_t *wkv_b, int B, float *out,
                  uint16_t *out_b16, int32_t *status, cudaStream_t s, bool pdl, const uint16_t *part_o = nullptr,
                  const float *part_lse = nullptr, int n_split = 0);

// Sparse attention (tensor-core kernel + split combine) over B query rows,
// T per sequence: row b is token b % T of cache sequence b / T, at position
// end_pos[b / T] - T + b % T, and sees the selected keys up to that position.
// Writes the normalised latent output o [B][128][512] as fp32 to o_out or as
// bf16 to o_b16 (exactly one non-NULL).  ws must hold attn_workspace(B, K)
// bytes (256-byte aligned).
// The split of the selection (n_split units per row, split_len entries each)
// depends on S_cap: caches of at most 65,535 rows stage 16-bit positions, so a
// unit holds up to 4096 entries instead of 2048.  The default S_cap gives the
// larger of the two workspaces, which covers every cache.
size_t attn_workspace(int B, int K, int *n_split = nullptr, int *split_len = nullptr, int S_cap = 1 << 30);
// With merge_later set and the selection split, the split-combine kernel is
// not launched: the partials stay in ws (attn_partials) for the consumer.
int launch_attn(const uint16_t *q_lat, const uint16_t *kv, const uint16_t *pe, int S_cap, const int32_t *topk, int K,
                const int32_t *end_pos, int B, int T, float softmax_scale, float *o_out, uint16_t *o_b16, void *ws,
                int32_t *status, cudaStream_t s, int *launches, bool merge_later = false);
// Where the split partials of launch_attn(B, K, S_cap) live in its workspace
// (part_o [B*n_split][128][512], fp32 -- bf16 when launched with merge_later --
// and part_lse [B*n_split][2][128]); n_split 1: none.
void attn_partials(int B, int K, int S_cap, void *ws, float **part_o, float **part_lse, int *n_split);

// Launch `kern` on stream s.  With pdl set, the launch allows programmatic
// dependent launch: the grid may be scheduled while the preceding grid of the
// stream is still running, and every kernel launched this way calls
// griddepcontrol.wait before it reads anything an earlier grid may write.
template <typename... KArgs, typename... Args>
cudaError_t launch_k(bool pdl, void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                     Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kern, static_cast<KArgs>(args)...);
}

// Raises kern's dynamic shared memory limit to `bytes` on the current device,
// once per device: the flag is atomic, so calls from several host threads are
// safe (two first calls may both set the attribute, which is harmless).
template <typename Kern>
bool smem_attr_once(std::atomic<bool> (&done)[64], Kern kern, int bytes) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return false;
    const bool cached = dev >= 0 && dev < 64;
    if (cached && done[dev].load(std::memory_order_acquire)) return true;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) != cudaSuccess) return false;
    if (cached) done[dev].store(true, std::memory_order_release);
    return true;
}

// TMA tensor map of a bf16 tensor (dims[0] innermost); false on failure.
bool make_tmap_bf16(CUtensorMap *map, const void *base, int rank, const uint64_t *dims,
                    const uint64_t *strides_bytes, const uint32_t *box, CUtensorMapSwizzle swizzle,
                    CUtensorMapL2promotion promotion = CU_TENSOR_MAP_L2_PROMOTION_L2_256B);

}  // namespace mla
