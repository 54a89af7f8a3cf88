// Commit of the accepted K/V rows, and prefill of cache rows, in the Q4_0 or
// the F16 cache format.
//
// "We got 207 tok/s with Qwen3.5-27B on an RTX 3090" (nowletus), "What we
// ported and tuned": Q4_0 KV cache; "Luce DFlash ..." (ai-navigate-news, ja),
// results paragraph: the F16 cache it is compared against. After greedy
// acceptance the accepted nodes' K/V rows are encoded into the cache at
// positions C .. C+L-1 and the committed length advances; rejected rows are
// never written.
//
// The commit moves at most (budget + 1) rows per KV head; it runs as one
// CTA so that reading C, writing the rows and advancing C need no
// inter-CTA ordering. One thread encodes one 32-value Q4_0 block, or eight
// values as binary16.

#include "common.cuh"

namespace dfv {

constexpr int kCommitThreads = 512;

struct CommitParams {
  int n_nodes, n_kv_heads, head_dim, capacity, fmt;
  int32_t* ctx_len;
  const int32_t* accept_len;
  const int32_t* path;
  const __nv_bfloat16* tree_k;
  const __nv_bfloat16* tree_v;
  uint8_t* k_cache;
  uint8_t* v_cache;
  uint32_t* status;
};

__device__ __forceinline__ void load_bf16_block(const __nv_bfloat16* src, float* x) {
  const uint4* v = reinterpret_cast<const uint4*>(src);   // 64 bytes, 16-byte aligned
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    const uint4 r = v[u];
    const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&r);
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float2 f = __bfloat1622float2(h[e]);
      x[u * 8 + 2 * e] = f.x;
      x[u * 8 + 2 * e + 1] = f.y;
    }
  }
}

__global__ void __launch_bounds__(kCommitThreads) commit_kernel(CommitParams p) {
  __shared__ int s_C, s_L, s_ok;
  __shared__ int s_path[kMaxNodes];
  if (threadIdx.x == 0) {
    const int C = *p.ctx_len, L = *p.accept_len;
    int ok = 1;
    if (C < 0 || C > p.capacity) { report(p.status, DFV_DEV_CTX); ok = 0; }
    else if (L < 1 || L > p.n_nodes) { report(p.status, DFV_DEV_BAD_PATH); ok = 0; }
    else if (C + L > p.capacity) { report(p.status, DFV_DEV_CAPACITY); ok = 0; }
    s_C = C;
    s_L = L;
    s_ok = ok;
  }
  __syncthreads();
  if (!s_ok) return;
  const int C = s_C, L = s_L;
  if (threadIdx.x < L) {
    const int node = p.path[threadIdx.x];
    if (node < 0 || node >= p.n_nodes) { s_ok = 0; report(p.status, DFV_DEV_BAD_PATH); }
    s_path[threadIdx.x] = node;
  }
  __syncthreads();
  if (!s_ok) return;
  const size_t row_bytes = static_cast<size_t>(kv_row_bytes(p.fmt, p.head_dim));
  if (p.fmt == DFV_KV_F16) {
    // eight values (16 bytes of bf16 -> 16 bytes of binary16) per item
    const int np = p.head_dim / 8;
    const int total = L * p.n_kv_heads * 2 * np;
    for (int it = threadIdx.x; it < total; it += kCommitThreads) {
      const int c = it % np;
      const int kv = (it / np) & 1;
      const int h = (it / (2 * np)) % p.n_kv_heads;
      const int k = it / (2 * np * p.n_kv_heads);
      const uint4 v = *reinterpret_cast<const uint4*>(
          (kv ? p.tree_v : p.tree_k) + (static_cast<size_t>(s_path[k]) * p.n_kv_heads + h) * p.head_dim + c * 8);
      *reinterpret_cast<uint4*>((kv ? p.v_cache : p.k_cache) +
                                (static_cast<size_t>(h) * p.capacity + C + k) * row_bytes + c * 16) =
          bf16x8_to_f16x8_rn(v);
    }
    __syncthreads();
    if (threadIdx.x == 0) *p.ctx_len = C + L;
    return;
  }
  const int nb = p.head_dim / 32;
  const int total = L * p.n_kv_heads * 2 * nb;
  for (int it = threadIdx.x; it < total; it += kCommitThreads) {
    const int b = it % nb;
    const int kv = (it / nb) & 1;
    const int h = (it / (2 * nb)) % p.n_kv_heads;
    const int k = it / (2 * nb * p.n_kv_heads);
    const __nv_bfloat16* src = (kv ? p.tree_v : p.tree_k) +
                               (static_cast<size_t>(s_path[k]) * p.n_kv_heads + h) * p.head_dim +
                               b * 32;
    float x[32];
    load_bf16_block(src, x);
    uint8_t* dst = (kv ? p.v_cache : p.k_cache) +
                   (static_cast<size_t>(h) * p.capacity + C + k) * row_bytes + b * 18;
    q4_0_quantize_block(x, dst);
  }
  __syncthreads();
  if (threadIdx.x == 0) *p.ctx_len = C + L;
}

struct QuantRowsParams {
  int n_kv_heads, head_dim, capacity, pos0, n_rows, fmt;
  const void* src;
  int64_t stride_row, stride_head;
  uint8_t* cache;
};

// F16 prefill: eight values per thread item, each rounded to binary16
// (nearest even).
template <typename T>
__global__ void __launch_bounds__(256) f16_rows_kernel(QuantRowsParams p) {
  const int np = p.head_dim / 8;
  const size_t row_bytes = static_cast<size_t>(p.head_dim) * 2;
  const int64_t total = static_cast<int64_t>(p.n_rows) * p.n_kv_heads * np;
  const T* src = static_cast<const T*>(p.src);
  for (int64_t it = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; it < total;
       it += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int c = static_cast<int>(it % np);
    const int h = static_cast<int>((it / np) % p.n_kv_heads);
    const int64_t r = it / (static_cast<int64_t>(np) * p.n_kv_heads);
    const T* s = src + r * p.stride_row + h * p.stride_head + c * 8;
    uint32_t w[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      float a, b;
      if constexpr (sizeof(T) == 4) { a = s[2 * k]; b = s[2 * k + 1]; }
      else { a = __bfloat162float(s[2 * k]); b = __bfloat162float(s[2 * k + 1]); }
      const __half2 hv = __floats2half2_rn(a, b);
      w[k] = *reinterpret_cast<const uint32_t*>(&hv);
    }
    *reinterpret_cast<uint4*>(p.cache + (static_cast<size_t>(h) * p.capacity + p.pos0 + r) * row_bytes +
                              c * 16) = make_uint4(w[0], w[1], w[2], w[3]);
  }
}

template <typename T>
__global__ void __launch_bounds__(256) quantize_rows_kernel(QuantRowsParams p) {
  const int nb = p.head_dim / 32;
  const size_t row_bytes = static_cast<size_t>(nb) * 18;
  const int64_t total = static_cast<int64_t>(p.n_rows) * p.n_kv_heads * nb;
  const T* src = static_cast<const T*>(p.src);
  for (int64_t it = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; it < total;
       it += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int b = static_cast<int>(it % nb);
    const int h = static_cast<int>((it / nb) % p.n_kv_heads);
    const int64_t r = it / (static_cast<int64_t>(nb) * p.n_kv_heads);
    const T* s = src + r * p.stride_row + h * p.stride_head + b * 32;
    float x[32];
#pragma unroll
    for (int k = 0; k < 32; ++k) {
      if constexpr (sizeof(T) == 4) x[k] = s[k];
      else x[k] = __bfloat162float(s[k]);
    }
    uint8_t* dst = p.cache + (static_cast<size_t>(h) * p.capacity + p.pos0 + r) * row_bytes + b * 18;
    q4_0_quantize_block(x, dst);
  }
}

dfv_status commit_launch(int n_nodes, int n_kv_heads, int head_dim, int kv_format,
                         int capacity, int32_t* ctx_len, const int32_t* accept_len,
                         const int32_t* path, const void* tree_k, const void* tree_v,
                         void* k_cache, void* v_cache, uint32_t* status, cudaStream_t stream) {
  if (kv_format != DFV_KV_Q4_0 && kv_format != DFV_KV_F16) return DFV_ERR_UNSUPPORTED;
  if (n_nodes < 1 || n_nodes > kMaxNodes || n_kv_heads < 1 || capacity < 0)
    return DFV_ERR_INVALID;
  if (head_dim != 64 && head_dim != 128 && head_dim != 256) return DFV_ERR_UNSUPPORTED;
  if (!ctx_len || !accept_len || !path || !tree_k || !tree_v || !k_cache || !v_cache)
    return DFV_ERR_INVALID;
  if (!aligned(tree_k, 16) || !aligned(tree_v, 16) || !aligned(k_cache, 16) ||
      !aligned(v_cache, 16))
    return DFV_ERR_INVALID;
  CommitParams p;
  p.n_nodes = n_nodes;
  p.n_kv_heads = n_kv_heads;
  p.head_dim = head_dim;
  p.capacity = capacity;
  p.fmt = kv_format;
  p.ctx_len = ctx_len;
  p.accept_len = accept_len;
  p.path = path;
  p.tree_k = static_cast<const __nv_bfloat16*>(tree_k);
  p.tree_v = static_cast<const __nv_bfloat16*>(tree_v);
  p.k_cache = static_cast<uint8_t*>(k_cache);
  p.v_cache = static_cast<uint8_t*>(v_cache);
  p.status = status;
  commit_kernel<<<1, kCommitThreads, 0, stream>>>(p);
  return cudaGetLastError() == cudaSuccess ? DFV_OK : DFV_ERR_CUDA;
}

}  // namespace dfv

extern "C" dfv_status dfv_kv_commit(int n_nodes, int n_kv_heads, int head_dim, int kv_format,
                                    int cache_capacity, int32_t* ctx_len,
                                    const int32_t* accept_len, const int32_t* path,
                                    const void* tree_k, const void* tree_v, void* k_cache,
                                    void* v_cache, uint32_t* status, dfv_stream_t stream) {
  return dfv::commit_launch(n_nodes, n_kv_heads, head_dim, kv_format, cache_capacity, ctx_len,
                            accept_len, path, tree_k, tree_v, k_cache, v_cache, status,
                            static_cast<cudaStream_t>(stream));
}

extern "C" dfv_status dfv_kv_quantize_rows(int n_kv_heads, int head_dim, int kv_format,
                                           int cache_capacity, int pos0, int n_rows,
                                           const void* src, int src_dtype, int64_t stride_row,
                                           int64_t stride_head, void* cache,
                                           dfv_stream_t stream) {
  using namespace dfv;
  if (kv_format != DFV_KV_Q4_0 && kv_format != DFV_KV_F16) return DFV_ERR_UNSUPPORTED;
  if (head_dim != 64 && head_dim != 128 && head_dim != 256) return DFV_ERR_UNSUPPORTED;
  if (src_dtype != DFV_DTYPE_F32 && src_dtype != DFV_DTYPE_BF16) return DFV_ERR_UNSUPPORTED;
  if (n_kv_heads < 1 || cache_capacity < 0 || pos0 < 0 || n_rows < 0 ||
      static_cast<int64_t>(pos0) + n_rows > cache_capacity)
    return DFV_ERR_INVALID;
  if (!src || !cache || !aligned(cache, 16)) return DFV_ERR_INVALID;
  if (n_rows == 0) return DFV_OK;
  QuantRowsParams p;
  p.n_kv_heads = n_kv_heads;
  p.head_dim = head_dim;
  p.capacity = cache_capacity;
  p.pos0 = pos0;
  p.n_rows = n_rows;
  p.fmt = kv_format;
  p.src = src;
  p.stride_row = stride_row;
  p.stride_head = stride_head;
  p.cache = static_cast<uint8_t*>(cache);
  const int per = kv_format == DFV_KV_F16 ? head_dim / 8 : head_dim / 32;   // thread items per row
  const int64_t total = static_cast<int64_t>(n_rows) * n_kv_heads * per;
  int64_t blocks = (total + 255) / 256;
  const int64_t cap = static_cast<int64_t>(sm_count()) * 16;
  if (blocks > cap) blocks = cap;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (kv_format == DFV_KV_F16) {
    if (src_dtype == DFV_DTYPE_F32)
      f16_rows_kernel<float><<<static_cast<int>(blocks), 256, 0, s>>>(p);
    else
      f16_rows_kernel<__nv_bfloat16><<<static_cast<int>(blocks), 256, 0, s>>>(p);
  } else if (src_dtype == DFV_DTYPE_F32) {
    quantize_rows_kernel<float><<<static_cast<int>(blocks), 256, 0, s>>>(p);
  } else {
    quantize_rows_kernel<__nv_bfloat16><<<static_cast<int>(blocks), 256, 0, s>>>(p);
  }
  return cudaGetLastError() == cudaSuccess ? DFV_OK : DFV_ERR_CUDA;
}
