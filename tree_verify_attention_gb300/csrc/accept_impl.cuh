// Kernel body of the per-node argmax + greedy walk (see accept.cu).
#pragma once

#include <climits>

#include "common.cuh"

namespace dfv {

constexpr int kAcceptThreads = 256;

// A (value, index) argmax partial (the fused step's logits slices).
struct ArgPartial {
  float v;
  int idx;
};

struct AcceptParams {
  int n_nodes, vocab, chunks, chunk_len;
  const void* logits;
  const int32_t* parent;
  const int32_t* tokens;
  int32_t* argmax;
  int32_t* accept_len;
  int32_t* path;
  int32_t* out_tokens;
  unsigned int* ticket;       // zero between launches
  unsigned long long* keys;   // [n_nodes] packed (value, index) maxima; zero between launches
  uint32_t* status;
};

// Workspace: the ticket in the first 256 bytes, then one 8-byte key per node.
constexpr size_t kAcceptHeaderBytes = 256;
inline size_t accept_scratch_bytes(int n_nodes) {
  return kAcceptHeaderBytes + ((static_cast<size_t>(n_nodes) * 8 + 255) & ~static_cast<size_t>(255));
}

// About four CTAs per SM over the whole grid, chunks of >= 2048 elements.
inline int accept_chunks(int n_nodes, int vocab) {
  const int sms = sm_count();
  const int want = (4 * sms + n_nodes - 1) / n_nodes;
  const int cap = (vocab + 2047) / 2048;
  int c = want < cap ? want : cap;
  return c < 1 ? 1 : c;
}

inline int accept_chunk_len(int vocab, int chunks) {
  const int c = (vocab + chunks - 1) / chunks;
  return (c + 7) & ~7;
}

// (v, i) beats (w, j): larger value, or equal value and lower index. -0.0
// and +0.0 compare equal, so the lower index wins between them.
__device__ __forceinline__ bool beats(float v, int i, float w, int j) {
  return v > w || (v == w && i < j);
}

// (value, index) packed so that the larger key is the winner under
// `beats`: the high word orders the floats (-0.0 taken as +0.0; every
// non-NaN value gives a high word of at least 0x007FFFFF, so a real key is
// above the zero a node's key starts from), the low word is ~index, larger
// for the lower index.
__device__ __forceinline__ unsigned long long arg_key(float v, int idx) {
  uint32_t b = __float_as_uint(v == 0.f ? 0.f : v);
  b = (b & 0x80000000u) ? ~b : (b | 0x80000000u);
  return (static_cast<unsigned long long>(b) << 32) | static_cast<uint32_t>(~static_cast<uint32_t>(idx));
}

__device__ __forceinline__ int key_index(unsigned long long k) {
  return static_cast<int>(~static_cast<uint32_t>(k));
}

__device__ __forceinline__ void warp_argmax(float& v, int& i) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float ov = __shfl_down_sync(0xffffffffu, v, o);
    const int oi = __shfl_down_sync(0xffffffffu, i, o);
    if (beats(ov, oi, v, i)) { v = ov; i = oi; }
  }
}

template <typename T>
__device__ __forceinline__ float to_f32(T x);
template <>
__device__ __forceinline__ float to_f32<float>(float x) { return x; }
template <>
__device__ __forceinline__ float to_f32<__nv_bfloat16>(__nv_bfloat16 x) {
  return __bfloat162float(x);
}

// Scan one 16-byte vector holding VE elements starting at index `base`,
// in increasing index order.
template <typename T>
__device__ __forceinline__ void scan_vec(const uint4& r, int base, float& best, int& bidx) {
  constexpr int VE = 16 / sizeof(T);
  const T* e = reinterpret_cast<const T*>(&r);
#pragma unroll
  for (int k = 0; k < VE; ++k) {
    const float v = to_f32<T>(e[k]);
    if (v > best || bidx == INT_MAX) { best = v; bidx = base + k; }
  }
}

// Merge per-thread (best, bidx) over a CTA of NT (<= 1024) threads; result
// valid in thread 0.
template <int NT = kAcceptThreads>
__device__ __forceinline__ void block_argmax(float& best, int& bidx) {
  __shared__ float sv[NT / 32];
  __shared__ int si[NT / 32];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  warp_argmax(best, bidx);
  if (lane == 0) { sv[warp] = best; si[warp] = bidx; }
  __syncthreads();
  if (warp == 0) {
    // the per-warp results merge in warp 0
    best = lane < NT / 32 ? sv[lane] : -INFINITY;
    bidx = lane < NT / 32 ? si[lane] : INT_MAX;
    warp_argmax(best, bidx);
  }
}

// Argmax of one row chunk [begin, end), per thread; elements of each
// thread are visited in increasing index order. U vectors per thread are in
// flight at once.
template <typename T, int U = 4, int NT = kAcceptThreads>
__device__ __forceinline__ void chunk_argmax(const T* row, int begin, int end, float& best,
                                             int& bidx) {
  constexpr int VE = 16 / sizeof(T);
  best = -INFINITY;
  bidx = INT_MAX;
  if (begin >= end) return;
  // scalar head up to a 16-byte boundary
  const uintptr_t addr = reinterpret_cast<uintptr_t>(row + begin);
  int head = static_cast<int>(((16 - (addr & 15)) & 15) / sizeof(T));
  if (head > end - begin) head = end - begin;
  const int tid = threadIdx.x;
  if (tid < head) {
    const float v = to_f32<T>(row[begin + tid]);
    best = v;
    bidx = begin + tid;
  }
  const int vbeg = begin + head;
  const int nvec = (end - vbeg) / VE;
  const uint4* vp = reinterpret_cast<const uint4*>(row + vbeg);
  for (int v0 = tid; v0 < nvec; v0 += U * NT) {
    uint4 r[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int v = v0 + u * NT;
      if (v < nvec) r[u] = __ldcs(vp + v);
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int v = v0 + u * NT;
      if (v < nvec) scan_vec<T>(r[u], vbeg + v * VE, best, bidx);
    }
  }
  // scalar tail
  const int tbeg = vbeg + nvec * VE;
  for (int k = tbeg + tid; k < end; k += NT) {
    const float v = to_f32<T>(row[k]);
    if (v > best || bidx == INT_MAX) { best = v; bidx = k; }
  }
}

// The walk, run by the last CTA once every node's key is final: one thread
// per node takes its key (and zeroes it for the next launch), then warp 0
// walks the tree with ballots and writes the outputs. `s_am` receives the
// argmax of every node.
__device__ __forceinline__ void accept_tail(const AcceptParams& p, int* s_am, int* s_path) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  // warp 0's tree loads go out first, beside the key exchanges below
  int par[3], tok[3];
  bool bad = false;
  if (warp == 0) {
#pragma unroll
    for (int s = 0; s < 3; ++s) {
      const int n = lane + 32 * s;
      par[s] = -2;
      tok[s] = 0;
      if (n >= 1 && n < p.n_nodes) {
        par[s] = p.parent[n];
        tok[s] = p.tokens[n];
      }
    }
  }
  for (int node = threadIdx.x; node < p.n_nodes; node += kAcceptThreads) {
    const int am = key_index(atomicExch(p.keys + node, 0ull));
    s_am[node] = am;
    p.argmax[node] = am;
  }
  if (threadIdx.x == 0) *p.ticket = 0u;   // ready for the next launch
  __syncthreads();
  if (warp != 0) return;
#pragma unroll
  for (int s = 0; s < 3; ++s) {
    const int n = lane + 32 * s;
    if (n >= 1 && n < p.n_nodes && (par[s] < 0 || par[s] >= n)) {
      bad = true;
      par[s] = 0;
    }
  }
  if (__any_sync(0xffffffffu, bad) && lane == 0) report(p.status, DFV_DEV_BAD_TREE);

  int cur = 0, L = 1;
  if (lane == 0) s_path[0] = 0;
  for (int it = 0; it < p.n_nodes; ++it) {
    const int t = s_am[cur];
    const unsigned b0 = __ballot_sync(0xffffffffu, par[0] == cur && tok[0] == t);
    const unsigned b1 = __ballot_sync(0xffffffffu, par[1] == cur && tok[1] == t);
    const unsigned b2 = __ballot_sync(0xffffffffu, par[2] == cur && tok[2] == t);
    int next = -1;
    if (b0) next = __ffs(b0) - 1;
    else if (b1) next = 31 + __ffs(b1);
    else if (b2) next = 63 + __ffs(b2);
    if (next < 0) break;
    if (lane == 0) s_path[L] = next;
    ++L;
    cur = next;
  }
  __syncwarp();
  for (int k = lane; k < p.n_nodes; k += 32) {
    p.path[k] = k < L ? s_path[k] : -1;
    int ot = -1;
    if (k < L - 1) ot = p.tokens[s_path[k + 1]];
    else if (k == L - 1) ot = s_am[s_path[L - 1]];
    p.out_tokens[k] = ot;
  }
  if (lane == 0) *p.accept_len = L;
}

// One CTA per (chunk, node): the chunk's argmax goes into the node's key by
// a 64-bit atomic max, then a ticket (release / acquire) counts the CTAs;
// the last one takes the keys and walks. No CTA waits for another.
template <typename T>
__global__ void __launch_bounds__(kAcceptThreads) accept_kernel(AcceptParams p) {
  __shared__ int s_am[kMaxNodes];
  __shared__ int s_path[kMaxNodes];
  __shared__ bool s_last;
  const int node = blockIdx.y, chunk = blockIdx.x;
  const int begin = chunk * p.chunk_len;
  const int end = min(p.vocab, begin + p.chunk_len);
  const T* row = static_cast<const T*>(p.logits) + static_cast<size_t>(node) * p.vocab;
  float best;
  int bidx;
  chunk_argmax<T>(row, begin, end, best, bidx);
  block_argmax(best, bidx);
  if (threadIdx.x == 0) {
    atomicMax(p.keys + node, arg_key(best, bidx));
    const unsigned total = gridDim.x * gridDim.y;
    unsigned int old;
    asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], 1;" : "=r"(old) : "l"(p.ticket) : "memory");
    s_last = old == total - 1;
  }
  __syncthreads();
  if (!s_last) return;
  accept_tail(p, s_am, s_path);
}

}  // namespace dfv
