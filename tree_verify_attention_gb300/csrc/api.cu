// Library-wide entry points: status strings, version, workspace clearing,
// device queries, and the whole verify step composed from the three parts.

#include <atomic>

#include "common.cuh"

namespace dfv {

// SMs of the current device, looked up once per device (an atomic per
// device: concurrent first lookups store the same value).
int sm_count() {
  static std::atomic<int> cached[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
  int n = cached[dev].load(std::memory_order_relaxed);
  if (n == 0) {
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
      n = 148;
    cached[dev].store(n, std::memory_order_relaxed);
  }
  return n;
}

size_t step_workspace_bytes(int n_nodes, int hq, int hkv, int head_dim, int window, int cap,
                            int vocab, bool with_accept);
dfv_status step_launch(bool with_accept, int n_nodes, int max_depth, int hq, int hkv,
                       int head_dim, int window, int kv_format, int cap, int vocab,
                       int logits_dtype, int32_t* ctx_len, void* k_cache, void* v_cache,
                       const void* q, const void* tree_k, const void* tree_v,
                       const int32_t* parent, const int32_t* tokens, const void* logits,
                       float scale, float* out, float* lse, int32_t* argmax, int32_t* accept_len,
                       int32_t* path, int32_t* out_tokens, void* workspace, size_t ws_bytes,
                       uint32_t* status, cudaStream_t stream);

}  // namespace dfv

extern "C" const char* dfv_status_string(dfv_status s) {
  switch (s) {
    case DFV_OK: return "ok";
    case DFV_ERR_INVALID: return "invalid argument";
    case DFV_ERR_UNSUPPORTED: return "unsupported configuration";
    case DFV_ERR_WORKSPACE: return "workspace too small";
    case DFV_ERR_CUDA: return "CUDA error";
  }
  return "unknown status";
}

extern "C" int dfv_version(void) { return 100; }

extern "C" dfv_status dfv_workspace_clear(void* workspace, size_t bytes, dfv_stream_t stream) {
  if (workspace == nullptr && bytes != 0) return DFV_ERR_INVALID;
  if (bytes == 0) return DFV_OK;
  return cudaMemsetAsync(workspace, 0, bytes, static_cast<cudaStream_t>(stream)) == cudaSuccess
             ? DFV_OK
             : DFV_ERR_CUDA;
}

extern "C" size_t dfv_tree_verify_attn_workspace_bytes(int n_nodes, int n_q_heads, int n_kv_heads,
                                                       int head_dim, int window,
                                                       int cache_capacity) {
  return dfv::step_workspace_bytes(n_nodes, n_q_heads, n_kv_heads, head_dim, window,
                                   cache_capacity, 0, false);
}

extern "C" dfv_status dfv_tree_verify_attn(int n_nodes, int max_depth, int n_q_heads,
                                           int n_kv_heads, int head_dim, int window,
                                           int kv_format, int cache_capacity,
                                           const int32_t* ctx_len, const void* k_cache,
                                           const void* v_cache, const void* q,
                                           const void* tree_k, const void* tree_v,
                                           const int32_t* parent, float scale, float* out,
                                           float* lse, void* workspace, size_t workspace_bytes,
                                           uint32_t* status, dfv_stream_t stream) {
  return dfv::step_launch(false, n_nodes, max_depth, n_q_heads, n_kv_heads, head_dim, window,
                          kv_format, cache_capacity, 0, 0, const_cast<int32_t*>(ctx_len),
                          const_cast<void*>(k_cache), const_cast<void*>(v_cache), q, tree_k,
                          tree_v, parent, nullptr, nullptr, scale, out, lse, nullptr, nullptr,
                          nullptr, nullptr, workspace, workspace_bytes, status,
                          static_cast<cudaStream_t>(stream));
}

extern "C" size_t dfv_verify_step_workspace_bytes(int n_nodes, int n_q_heads, int n_kv_heads,
                                                  int head_dim, int window, int cache_capacity,
                                                  int vocab) {
  return dfv::step_workspace_bytes(n_nodes, n_q_heads, n_kv_heads, head_dim, window,
                                   cache_capacity, vocab, true);
}

extern "C" int dfv_verify_step_launches(int n_nodes, int n_q_heads, int n_kv_heads, int head_dim,
                                        int window, int cache_capacity) {
  return dfv::step_workspace_bytes(n_nodes, n_q_heads, n_kv_heads, head_dim, window,
                                   cache_capacity, 1, true) ? 1 : -1;
}

extern "C" dfv_status dfv_verify_step(int n_nodes, int max_depth, int n_q_heads, int n_kv_heads,
                                      int head_dim, int window, int kv_format,
                                      int cache_capacity, int vocab, int logits_dtype,
                                      int32_t* ctx_len, void* k_cache, void* v_cache,
                                      const void* q, const void* tree_k, const void* tree_v,
                                      const int32_t* parent, const int32_t* tokens,
                                      const void* logits, float scale, float* out, float* lse,
                                      int32_t* argmax, int32_t* accept_len, int32_t* path,
                                      int32_t* out_tokens, void* workspace,
                                      size_t workspace_bytes, uint32_t* status,
                                      dfv_stream_t stream) {
  return dfv::step_launch(true, n_nodes, max_depth, n_q_heads, n_kv_heads, head_dim, window,
                          kv_format, cache_capacity, vocab, logits_dtype, ctx_len, k_cache,
                          v_cache, q, tree_k, tree_v, parent, tokens, logits, scale, out, lse,
                          argmax, accept_len, path, out_tokens, workspace, workspace_bytes,
                          status, static_cast<cudaStream_t>(stream));
}
