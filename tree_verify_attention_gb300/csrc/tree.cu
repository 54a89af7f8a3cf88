// Draft-tree bookkeeping as a standalone entry point: the depth of every
// node and its ancestor-or-self bitmask, the tree half of the visibility
// rule of the tree-verify attention ("Luce DFlash: Qwen3.6-27B ..."
// (ai-navigate-news, ja), feature list: DDTree tree-verify; a node attends
// to its ancestors and itself). The step kernel computes the same values
// internally; this is for callers that build their own masks.
//
// One CTA of kTreeThreads threads, one node per thread, by pointer jumping
// in shared memory: after round r, J[i] is the (2^r)-th ancestor of i (or
// -1 past the root), D[i] the distance to it, and A[i] the set of nodes on
// the path from i up to (excluding) J[i]. ceil(log2 N) rounds reach past
// every root path (depth < N).

#include "common.cuh"

namespace dfv {

constexpr int kTreeThreads = ((kMaxNodes + 31) / 32) * 32;   // 96
static_assert(kMaskWords == DFV_MASK_WORDS, "mask words");

__global__ void __launch_bounds__(kTreeThreads) tree_mask_kernel(int n, const int32_t* parent,
                                                                 int32_t* depth, uint32_t* anc,
                                                                 uint32_t* status) {
  __shared__ int sJ[kMaxNodes], sD[kMaxNodes];
  __shared__ uint32_t sA[kMaxNodes][kMaskWords];
  const int t = threadIdx.x;
  if (t < n) {
    int pa = t == 0 ? -1 : parent[t];
    if (t > 0 && (pa < 0 || pa >= t)) {
      report(status, DFV_DEV_BAD_TREE);
      pa = 0;
    }
    sJ[t] = pa;
    sD[t] = t > 0 ? 1 : 0;
#pragma unroll
    for (int w = 0; w < kMaskWords; ++w) sA[t][w] = (t >> 5) == w ? (1u << (t & 31)) : 0u;
  }
  __syncthreads();
  int rounds = 0;
  while ((1 << rounds) < n) ++rounds;
#pragma unroll 1
  for (int round = 0; round < rounds; ++round) {
    int j = -1, nd = 0, nj = -1;
    uint32_t nm[kMaskWords];
    if (t < n) {
      j = sJ[t];
      if (j >= 0) {
        nd = sD[t] + sD[j];
        nj = sJ[j];
#pragma unroll
        for (int w = 0; w < kMaskWords; ++w) nm[w] = sA[t][w] | sA[j][w];
      }
    }
    __syncthreads();
    if (t < n && j >= 0) {
      sD[t] = nd;
      sJ[t] = nj;
#pragma unroll
      for (int w = 0; w < kMaskWords; ++w) sA[t][w] = nm[w];
    }
    __syncthreads();
  }
  if (t < n) {
    depth[t] = sD[t];
#pragma unroll
    for (int w = 0; w < kMaskWords; ++w) anc[t * kMaskWords + w] = sA[t][w];
  }
}

}  // namespace dfv

extern "C" dfv_status dfv_build_tree_mask(int n_nodes, const int32_t* parent, int32_t* depth,
                                          uint32_t* anc_mask, uint32_t* status,
                                          dfv_stream_t stream) {
  if (n_nodes < 1 || n_nodes > DFV_MAX_NODES || parent == nullptr || depth == nullptr ||
      anc_mask == nullptr)
    return DFV_ERR_INVALID;
  dfv::tree_mask_kernel<<<1, dfv::kTreeThreads, 0, static_cast<cudaStream_t>(stream)>>>(
      n_nodes, parent, depth, anc_mask, status);
  return cudaGetLastError() == cudaSuccess ? DFV_OK : DFV_ERR_CUDA;
}
