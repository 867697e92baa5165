// mla_sparse_decode_static_ws: the same decode as mla_sparse_decode, for
// callers that cannot allocate device memory themselves.
//
// Some callers have no allocator to draw from: plugin hosts that own every
// device buffer and give extensions only the tensors they pass in,
// latency-critical serving loops that forbid allocator calls (a cudaMalloc
// may synchronise the device), and code whose memory plan is fixed ahead of
// time.  They can still hand over inputs and outputs, but not a workspace.
// This entry point takes its scratch from one fixed array that lives in this
// library's device image instead.
#include "common.cuh"
#include "kernels.cuh"

#include <mutex>

namespace {

// Scratch shared by every call of mla_sparse_decode_static_ws on a device.
// It is part of the library's device image: each GPU that loads the library
// keeps these MLA_STATIC_WS_BYTES reserved until the process exits.
static __device__ __align__(256) unsigned char g_static_ws[MLA_STATIC_WS_BYTES];

// Device address of g_static_ws per device.  The name g_static_ws in host
// code is only a host-side stand-in, so the address is looked up once per
// device, with that device current.
struct StaticWsAddr {
    std::mutex mu;
    void *ptr[64] = {};
};

StaticWsAddr &addr_table() {
    static StaticWsAddr t;
    return t;
}

int static_ws_ptr(void **out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return MLA_ERR_CUDA;
    if (dev < 0 || dev >= 64) return MLA_ERR_DEVICE;
    StaticWsAddr &t = addr_table();
    std::lock_guard<std::mutex> lock(t.mu);
    if (!t.ptr[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_static_ws) != cudaSuccess || !p) return MLA_ERR_CUDA;
        t.ptr[dev] = p;
    }
    *out = t.ptr[dev];
    return MLA_OK;
}

}  // namespace

extern "C" int mla_sparse_decode_static_ws(const mla_bf16 *q_lat, const mla_bf16 *kv_cache, const mla_bf16 *pe_cache,
                                           int S_cap, const int32_t *topk_idx, int K, const int32_t *end_pos, int B,
                                           float softmax_scale, const mla_bf16 *wkv_b, float *out,
                                           int32_t *dev_status, mla_stream_t stream) {
    const size_t need = mla_sparse_decode_workspace_size(B, K);
    if (need == 0 || need > MLA_STATIC_WS_BYTES) return MLA_ERR_SIZE;
    void *ws = nullptr;
    const int rc = static_ws_ptr(&ws);
    if (rc != MLA_OK) return rc;
    // nothing in the scratch has to start at zero: every byte the kernels read
    // is written earlier in the same call
    return mla_sparse_decode(q_lat, kv_cache, pe_cache, S_cap, topk_idx, K, end_pos, B, softmax_scale, wkv_b, out, ws,
                             MLA_STATIC_WS_BYTES, dev_status, stream);
}
