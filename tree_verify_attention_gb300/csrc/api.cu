// Library-wide entry points: status strings, version, workspace clearing,
// device queries, and the whole verify step composed from the three parts.

#include "common.cuh"

namespace dfv {

int sm_count() {
  static int cached[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
  if (cached[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
      n = 148;
    cached[dev] = n;
  }
  return cached[dev];
}

size_t attn_workspace_bytes(int n_nodes, int hq, int hkv, int head_dim, int window, int cap);
dfv_status attn_launch(int n_nodes, int max_depth, int hq, int hkv, int head_dim, int window,
                       int kv_format, int cap, const int32_t* ctx_len, const void* k_cache,
                       const void* v_cache, const void* q, const void* tree_k,
                       const void* tree_v, const int32_t* parent, float scale, float* out,
                       float* lse, void* workspace, size_t ws_bytes, uint32_t* status,
                       cudaStream_t stream);
int attn_launches(int n_nodes, int hq, int hkv, int head_dim, int window, int cap);
size_t accept_workspace_bytes(int n_nodes, int vocab);
dfv_status accept_launch(int n_nodes, int vocab, int dtype, const void* logits,
                         const int32_t* parent, const int32_t* tokens, int32_t* argmax,
                         int32_t* accept_len, int32_t* path, int32_t* out_tokens,
                         void* workspace, size_t ws_bytes, uint32_t* status,
                         cudaStream_t stream);
dfv_status commit_launch(int n_nodes, int n_kv_heads, int head_dim, int kv_format,
                         int capacity, int32_t* ctx_len, const int32_t* accept_len,
                         const int32_t* path, const void* tree_k, const void* tree_v,
                         void* k_cache, void* v_cache, uint32_t* status, cudaStream_t stream);

static size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

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

extern "C" size_t dfv_verify_step_workspace_bytes(int n_nodes, int n_q_heads, int n_kv_heads,
                                                  int head_dim, int window, int cache_capacity,
                                                  int vocab) {
  const size_t a = dfv::accept_workspace_bytes(n_nodes, vocab);
  const size_t b = dfv::attn_workspace_bytes(n_nodes, n_q_heads, n_kv_heads, head_dim, window,
                                             cache_capacity);
  if (a == 0 || b == 0) return 0;
  return dfv::align256(a) + b;
}

extern "C" int dfv_verify_step_launches(int n_nodes, int n_q_heads, int n_kv_heads, int head_dim,
                                        int window, int cache_capacity) {
  const int a = dfv::attn_launches(n_nodes, n_q_heads, n_kv_heads, head_dim, window,
                                   cache_capacity);
  return a < 0 ? -1 : a + 2;   // attention (+ merge), argmax + walk, commit
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
  using namespace dfv;
  if (n_nodes < 1 || n_nodes > kMaxNodes || vocab < 1) return DFV_ERR_INVALID;
  const size_t need = dfv_verify_step_workspace_bytes(n_nodes, n_q_heads, n_kv_heads, head_dim,
                                                      window, cache_capacity, vocab);
  if (need == 0) return DFV_ERR_INVALID;
  if (workspace == nullptr || !aligned(workspace, 256)) return DFV_ERR_INVALID;
  if (workspace_bytes < need) return DFV_ERR_WORKSPACE;
  // everything the later launches check, checked before the first launch
  if (logits_dtype != DFV_DTYPE_F32 && logits_dtype != DFV_DTYPE_BF16) return DFV_ERR_UNSUPPORTED;
  if (!logits || !tokens || !argmax || !accept_len || !path || !out_tokens) return DFV_ERR_INVALID;
  const size_t a = align256(accept_workspace_bytes(n_nodes, vocab));
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  dfv_status st = attn_launch(n_nodes, max_depth, n_q_heads, n_kv_heads, head_dim, window,
                              kv_format, cache_capacity, ctx_len, k_cache, v_cache, q, tree_k,
                              tree_v, parent, scale, out, lse, static_cast<char*>(workspace) + a,
                              workspace_bytes - a, status, s);
  if (st != DFV_OK) return st;
  st = accept_launch(n_nodes, vocab, logits_dtype, logits, parent, tokens, argmax, accept_len,
                     path, out_tokens, workspace, a, status, s);
  if (st != DFV_OK) return st;
  return commit_launch(n_nodes, n_kv_heads, head_dim, kv_format, cache_capacity, ctx_len,
                       accept_len, path, tree_k, tree_v, k_cache, v_cache, status, s);
}
