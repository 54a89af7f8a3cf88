// dfv_greedy_accept_static: the per-node argmax + greedy walk of
// dfv_greedy_accept, with its scratch in a fixed device array inside this
// library instead of a caller-provided workspace.
//
// Who needs it: callers that cannot allocate device memory where they
// verify. A plugin inside a serving framework that owns every device
// allocation is handed only its input and output buffers and has no
// allocator to ask for scratch; a latency-critical decode loop cannot
// afford cudaMalloc / cudaFree there, because they may synchronise the
// whole device and stall every other stream. Such callers pass inputs and
// outputs only; this file supplies the scratch.
//
// The array (kStaticBytes) is a file-scope __device__ variable: every GPU
// that loads the library holds it until the process exits. Host code cannot
// use its name as a device address, so the first call on each device looks
// its address up with cudaGetSymbolAddress (with that device current) and
// caches it (an atomic per device, so host threads making their first
// calls at once agree on it). That first call may also load the module on
// the device, so it should happen before any stream capture. The cached
// address belongs to the device's current context: after cudaDeviceReset
// the library must not be used again in the process. Every call on a device
// uses the same array; calls whose kernels overlap on the GPU race on it.

#include <atomic>

#include "common.cuh"
#include "accept_impl.cuh"

namespace dfv {

constexpr size_t kStaticBytes = DFV_GREEDY_ACCEPT_STATIC_SCRATCH_BYTES;

static __device__ __align__(256) unsigned char g_accept_scratch[kStaticBytes];

size_t accept_workspace_bytes(int n_nodes, int vocab);

namespace {

constexpr int kMaxDevices = 64;
std::atomic<void*> g_scratch_ptr[kMaxDevices];

// Address of this device's array, looked up once per device. Two threads
// racing on the first lookup both get the same address from the runtime,
// so either store is correct.
void* scratch_for_current_device() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  void* p = g_scratch_ptr[dev].load(std::memory_order_acquire);
  if (p == nullptr) {
    if (cudaGetSymbolAddress(&p, g_accept_scratch) != cudaSuccess) return nullptr;
    g_scratch_ptr[dev].store(p, std::memory_order_release);
  }
  return p;
}

}  // namespace
}  // namespace dfv

extern "C" dfv_status dfv_greedy_accept_static(int n_nodes, int vocab, int logits_dtype,
                                               const void* logits, const int32_t* parent,
                                               const int32_t* tokens, int32_t* argmax,
                                               int32_t* accept_len, int32_t* path,
                                               int32_t* out_tokens, uint32_t* status,
                                               dfv_stream_t stream) {
  using namespace dfv;
  if (n_nodes < 1 || n_nodes > kMaxNodes || vocab < 1) return DFV_ERR_INVALID;
  if (logits_dtype != DFV_DTYPE_F32 && logits_dtype != DFV_DTYPE_BF16) return DFV_ERR_UNSUPPORTED;
  if (!logits || !parent || !tokens || !argmax || !accept_len || !path || !out_tokens)
    return DFV_ERR_INVALID;
  // the problem must fit the fixed array
  if (accept_workspace_bytes(n_nodes, vocab) > kStaticBytes) return DFV_ERR_WORKSPACE;
  void* scratch = scratch_for_current_device();
  if (scratch == nullptr) return DFV_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // The array keeps whatever the previous call left; the ticket and the keys
  // must start at zero, so clear them in stream order before the kernel.
  if (cudaMemsetAsync(scratch, 0, accept_scratch_bytes(n_nodes), s) != cudaSuccess) return DFV_ERR_CUDA;
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
  p.ticket = reinterpret_cast<unsigned int*>(scratch);
  p.keys = reinterpret_cast<unsigned long long*>(static_cast<char*>(scratch) + kAcceptHeaderBytes);
  p.status = status;
  dim3 grid(chunks, n_nodes);
  if (logits_dtype == DFV_DTYPE_BF16)
    accept_kernel<__nv_bfloat16><<<grid, kAcceptThreads, 0, s>>>(p);
  else
    accept_kernel<float><<<grid, kAcceptThreads, 0, s>>>(p);
  return cudaGetLastError() == cudaSuccess ? DFV_OK : DFV_ERR_CUDA;
}
