// Per-node vocabulary argmax + greedy tree walk, one launch.
//
// "Luce DFlash: Qwen3.6-27B ..." (ai-navigate-news, ja), feature list and
// constraints paragraph: verification is greedy only. The target token of a
// tree node is the argmax of its logits (lowest index on ties); the walk
// accepts, from the root, the lowest-index child whose draft token equals
// the last accepted node's target token, until none does.
//
// Design: the logits stream is HBM-bound (151936 x 23 bf16 = 7 MB per
// step), so each (node, chunk) CTA streams its chunk with 16-byte loads,
// all issued before any compare, and folds its (value, index) maximum into
// the node's 64-bit key with one atomic max (the packing makes the larger
// key the larger value, then the lower index). The last CTA to finish
// (atomic ticket in the workspace) exchanges each node's key for zero and
// runs the walk in one warp: ballots pick the lowest matching child. Keys
// and ticket end at zero, so the workspace stays zeroed.

#include "common.cuh"
#include "accept_impl.cuh"

namespace dfv {

size_t accept_workspace_bytes(int n_nodes, int /*vocab*/) {
  return accept_scratch_bytes(n_nodes);
}

dfv_status accept_launch(int n_nodes, int vocab, int dtype, const void* logits,
                         const int32_t* parent, const int32_t* tokens, int32_t* argmax,
                         int32_t* accept_len, int32_t* path, int32_t* out_tokens,
                         void* workspace, size_t ws_bytes, uint32_t* status,
                         cudaStream_t stream) {
  if (n_nodes < 1 || n_nodes > kMaxNodes || vocab < 1) return DFV_ERR_INVALID;
  if (dtype != DFV_DTYPE_F32 && dtype != DFV_DTYPE_BF16) return DFV_ERR_UNSUPPORTED;
  if (!logits || !parent || !tokens || !argmax || !accept_len || !path || !out_tokens ||
      !workspace)
    return DFV_ERR_INVALID;
  if (!aligned(workspace, 256)) return DFV_ERR_INVALID;
  if (ws_bytes < accept_workspace_bytes(n_nodes, vocab)) return DFV_ERR_WORKSPACE;
  const int chunks = accept_chunks(n_nodes, vocab);
  AcceptParams p;
  p.n_nodes = n_nodes;
  p.vocab = vocab;
  p.chunks = chunks;
  p.chunk_len = accept_chunk_len(vocab, chunks);
  p.logits = logits;
  p.parent = parent;
  p.tokens = tokens;
  p.argmax = argmax;
  p.accept_len = accept_len;
  p.path = path;
  p.out_tokens = out_tokens;
  p.ticket = reinterpret_cast<unsigned int*>(workspace);
  p.keys = reinterpret_cast<unsigned long long*>(static_cast<char*>(workspace) + kAcceptHeaderBytes);
  p.status = status;
  dim3 grid(chunks, n_nodes);
  if (dtype == DFV_DTYPE_BF16)
    accept_kernel<__nv_bfloat16><<<grid, kAcceptThreads, 0, stream>>>(p);
  else
    accept_kernel<float><<<grid, kAcceptThreads, 0, stream>>>(p);
  return cudaGetLastError() == cudaSuccess ? DFV_OK : DFV_ERR_CUDA;
}

}  // namespace dfv

extern "C" size_t dfv_greedy_accept_workspace_bytes(int n_nodes, int vocab) {
  if (n_nodes < 1 || n_nodes > dfv::kMaxNodes || vocab < 1) return 0;
  return dfv::accept_workspace_bytes(n_nodes, vocab);
}

extern "C" dfv_status dfv_greedy_accept(int n_nodes, int vocab, int logits_dtype,
                                        const void* logits, const int32_t* parent,
                                        const int32_t* tokens, int32_t* argmax,
                                        int32_t* accept_len, int32_t* path,
                                        int32_t* out_tokens, void* workspace,
                                        size_t workspace_bytes, uint32_t* status,
                                        dfv_stream_t stream) {
  return dfv::accept_launch(n_nodes, vocab, logits_dtype, logits, parent, tokens, argmax,
                            accept_len, path, out_tokens, workspace, workspace_bytes, status,
                            static_cast<cudaStream_t>(stream));
}
