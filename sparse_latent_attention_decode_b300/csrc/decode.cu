// mla_sparse_decode: sparse latent attention (attn.cu) followed, when wkv_b is
// given, by the value up-projection (out_up.cu); workspace layout and the
// host-side argument checks of the entry point.
//
// Source: DeepSeek-V3.2-Exp atlas, "Attention weights" page, excerpt
// mla-decode (scores, selection mask, softmax, PV, up-projection).
#include "common.cuh"
#include "kernels.cuh"

#include <atomic>
#include <cstring>
#include <mutex>

namespace mla {

struct WsLayout {
    size_t attn, o_lat, total;
};

static inline size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

static WsLayout ws_layout(int B, int K) {
    WsLayout w{};
    w.attn = 0;
    w.o_lat = align256(attn_workspace(B, K));
    w.total = w.o_lat + align256((size_t)B * H * C * sizeof(uint16_t));   // bf16 o for the up-projection
    return w;
}

}  // namespace mla

namespace mla {
static std::atomic<uint64_t> g_wait_limit_ns{2000000000ull};
uint64_t wait_limit_ns() { return g_wait_limit_ns.load(std::memory_order_relaxed); }
}  // namespace mla

using namespace mla;

extern "C" uint64_t mla_set_wait_limit_ns(uint64_t ns) {
    return g_wait_limit_ns.exchange(ns == 0 ? 1ull : ns);
}

extern "C" size_t mla_sparse_decode_workspace_size(int B, int K) {
    if (B < 1 || B > 4096 || K < 1 || K > (1 << 20)) return 0;
    return ws_layout(B, K).total;
}

extern "C" int mla_sparse_decode_tokens(const mla_bf16 *q_lat, const mla_bf16 *kv_cache, const mla_bf16 *pe_cache,
                                        int S_cap, const int32_t *topk_idx, int K, const int32_t *end_pos, int n_seq,
                                        int T, float softmax_scale, const mla_bf16 *wkv_b, void *out, int out_bf16,
                                        void *workspace, size_t ws_bytes, int32_t *dev_status, mla_stream_t stream) {
    if (!q_lat || !kv_cache || !pe_cache || !topk_idx || !end_pos || !out || !workspace) return MLA_ERR_NULL;
    if (!aligned16(q_lat) || !aligned16(kv_cache) || !aligned16(pe_cache) || !aligned16(topk_idx) ||
        !aligned16(out) || (wkv_b && !aligned16(wkv_b)) || (reinterpret_cast<uintptr_t>(workspace) & 255u))
        return MLA_ERR_ALIGN;
    if (n_seq < 1 || T < 1 || (long long)n_seq * T > 4096 || K < 1 || K > (1 << 20) || S_cap < 1 ||
        (long long)n_seq * S_cap >= (1ll << 31) || (out_bf16 != 0 && out_bf16 != 1))
        return MLA_ERR_SIZE;
    const int B = n_seq * T;   // query rows
    const WsLayout L = ws_layout(B, K);
    if (ws_bytes < L.total) return MLA_ERR_WORKSPACE;
    cudaStream_t s = (cudaStream_t)stream;
    char *ws = static_cast<char *>(workspace);
    // with wkv_b the latent output stays internal, as bf16 (the up-projection
    // rounds its operand to bf16 anyway); without it, o is the fp32 result
    float *out_f32 = out_bf16 ? nullptr : static_cast<float *>(out);
    uint16_t *out_b16 = out_bf16 ? static_cast<uint16_t *>(out) : nullptr;
    // with wkv_b the latent o goes through the workspace (bf16) to the up-projection
    uint16_t *o_b16 = wkv_b ? reinterpret_cast<uint16_t *>(ws + L.o_lat) : out_b16;
    int launches = 0;
    // With wkv_b, one or two query rows and a split selection, the
    // up-projection merges the split partials itself: no combine kernel and no
    // bf16 o round trip, which at this size is mostly launch latency.  With
    // more rows each up-projection CTA (one per head) would merge many rows in
    // turn, and the parallel combine kernel is faster (measured at B = 16, 32).
    const bool merge_in_up = wkv_b && B <= 2;
    int rc = launch_attn(q_lat, kv_cache, pe_cache, S_cap, topk_idx, K, end_pos, B, T, softmax_scale,
                         wkv_b ? nullptr : out_f32, o_b16, ws + L.attn, dev_status, s, &launches, merge_in_up);
    count_launches(launches);
    if (rc != MLA_OK) return rc;
    const ProfileHook &hook = profile_hook();
    const bool pdl = !(hook.start && hook.stop);
    if (wkv_b) {
        float *part_o = nullptr, *part_lse = nullptr;
        int n_split = 1;
        attn_partials(B, K, S_cap, ws + L.attn, &part_o, &part_lse, &n_split);
        if (merge_in_up && n_split > 1)
            return launch_out_up(nullptr, nullptr, wkv_b, B, out_f32, out_b16, dev_status, s, pdl,
                                 reinterpret_cast<const uint16_t *>(part_o), part_lse, n_split);
        return launch_out_up(nullptr, o_b16, wkv_b, B, out_f32, out_b16, dev_status, s, pdl);
    }
    return MLA_OK;
}

extern "C" int mla_sparse_decode(const mla_bf16 *q_lat, const mla_bf16 *kv_cache, const mla_bf16 *pe_cache,
                                 int S_cap, const int32_t *topk_idx, int K, const int32_t *end_pos, int B,
                                 float softmax_scale, const mla_bf16 *wkv_b, float *out, void *workspace,
                                 size_t ws_bytes, int32_t *dev_status, mla_stream_t stream) {
    return mla_sparse_decode_tokens(q_lat, kv_cache, pe_cache, S_cap, topk_idx, K, end_pos, B, 1, softmax_scale,
                                    wkv_b, out, 0, workspace, ws_bytes, dev_status, stream);
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
    if (code > 0 && code < 32) {
        // one description per combination of the MLA_DEV_* bits
        static const char *bit_names[5] = {"bad end_pos", "position outside rotary table", "on-chip wait timed out",
                                           "partial score outside the exchange range",
                                           "repeated position in a selection row"};
        static char names[32][208];
        static std::once_flag once;
        std::call_once(once, [] {
            for (int c = 1; c < 32; ++c) {
                names[c][0] = 0;
                for (int i = 0; i < 5; ++i) {
                    if (!(c & (1 << i))) continue;
                    if (names[c][0]) strcat(names[c], "; ");
                    strcat(names[c], bit_names[i]);
                }
            }
        });
        return names[code];
    }
    return "unknown status code";
}
