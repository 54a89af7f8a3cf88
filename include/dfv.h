/*
 * dfv.h -- C ABI of libdfv, the greedy DDTree tree-verify step on GB300
 * (sm_103a).
 *
 * The step (as described on "Luce DFlash: Qwen3.6-27B aiming for up to 2x
 * throughput on a single RTX 3090", ai-navigate-news (ja), feature list:
 * DDTree tree-verify, block size 16, default budget 22, greedy
 * verification, Q4_0 KV cache, 2048-token sliding-window flash attention at
 * decode; and "We got 207 tok/s with Qwen3.5-27B on an RTX 3090", nowletus,
 * DFlash section) has four parts, one entry point each:
 *
 *   dfv_tree_verify_attn  tree-masked attention of the N = budget + 1 draft
 *                         nodes over the Q4_0 cache (dequantised on the fly)
 *   dfv_greedy_accept     per-node vocabulary argmax + greedy tree walk
 *   dfv_kv_commit         Q4_0 re-quantisation of the accepted K/V rows into
 *                         the cache; rejected rows are never written
 *   dfv_verify_step       the three above in one launch
 *
 * plus dfv_kv_quantize_rows, the same Q4_0 quantiser used to fill a cache
 * from float rows (prefill).
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * - All tensor pointers are DEVICE pointers owned by the caller. The library
 *   allocates no memory. Scratch memory ("workspace") is passed in by the
 *   caller; its size comes from the matching *_workspace_bytes() query.
 * - Calls are asynchronous on `stream` (a cudaStream_t passed as void*;
 *   NULL = the legacy default stream). No entry point synchronises.
 * - The return value reports only what the host can check before launch:
 *   DFV_ERR_INVALID (null pointer, size out of range, misaligned pointer),
 *   DFV_ERR_UNSUPPORTED (valid but unsupported combination),
 *   DFV_ERR_WORKSPACE (workspace too small), DFV_ERR_CUDA (launch failed;
 *   the CUDA error is left for the caller to read). Nothing is launched when
 *   an error is returned.
 * - Problems only the device can see are OR-ed into `*status` (a device
 *   uint32, may be NULL): DFV_DEV_* bits below. The caller clears it.
 * - The committed length lives in device memory (`ctx_len`), so a loop of
 *   steps never needs a host round trip.
 * - bf16 / f16 / f32 are IEEE types in little-endian device memory.
 *
 * Data layouts
 * ------------
 * KV cache (K and V each), kv_format DFV_KV_Q4_0: Q4_0 blocks,
 *   [n_kv_heads][cache_capacity][D/32], one block = 18 bytes: fp16 scale d,
 *   then 16 bytes of 4-bit codes (byte j = code j in the low nibble, code
 *   j+16 in the high nibble); the block's values are (code - 8) * d. Row
 *   (head h, position p) starts at byte (h * cache_capacity + p) * (D / 32)
 *   * 18. Base pointer 16-byte aligned.
 * KV cache, kv_format DFV_KV_F16 ("Luce DFlash ..." results paragraph: the
 *   F16 cache that Q4_0 is compared against): binary16 values,
 *   [n_kv_heads][cache_capacity][D], row (h, p) at byte
 *   (h * cache_capacity + p) * D * 2; written with round-to-nearest-even.
 * Tree nodes: node 0 is the root; parent[i] in [0, i) for i >= 1 (parent[0]
 *   is ignored). Committed key j sits at position j, node i at position
 *   ctx_len + depth(i).
 * Visibility: node i sees committed key j iff j < ctx_len and
 *   (window == 0 or ctx_len + depth(i) - j < window), and tree node t iff t
 *   is i or an ancestor of i. Query head h uses KV head h / (Hq / Hkv).
 */
#ifndef DFV_H
#define DFV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef void* dfv_stream_t; /* a cudaStream_t */

typedef enum dfv_status {
  DFV_OK = 0,
  DFV_ERR_INVALID = 1,
  DFV_ERR_UNSUPPORTED = 2,
  DFV_ERR_WORKSPACE = 3,
  DFV_ERR_CUDA = 4
} dfv_status;

/* Device-detected problems, OR-ed into *status. */
#define DFV_DEV_BAD_TREE 0x1u  /* parent[i] outside [0, i): treated as 0      */
#define DFV_DEV_DEPTH 0x2u     /* a node deeper than max_depth (still run)    */
#define DFV_DEV_CAPACITY 0x4u  /* ctx_len + accept_len > capacity: no write   */
#define DFV_DEV_CTX 0x8u       /* *ctx_len outside [0, capacity]: nothing    */
                               /* committed; attention uses it clamped       */
#define DFV_DEV_BAD_PATH 0x10u /* path entry outside [0, n_nodes): no write   */
#define DFV_DEV_TIMEOUT 0x20u  /* a bounded wait gave up; outputs undefined   */
/* Every wait of a kernel (on a copy, an MMA, or another CTA of the step)
 * gives up after 100 ms of the GPU's global timer and sets DFV_DEV_TIMEOUT;
 * the kernel then skips what depended on the wait (a walker that timed out
 * commits nothing) and returns. Clear the workspace (dfv_workspace_clear)
 * before using it again after a timeout. */

#define DFV_KV_F16 1  /* binary16 values, 2 * D bytes per row                */
#define DFV_KV_Q4_0 2 /* Q4_0 blocks, D / 32 * 18 bytes per row               */
/* Flag OR-ed into kv_format of the attention entry points: attend the tree
 * nodes' K/V as the commit stores them in the cache format (Q4_0: quantised
 * and dequantised; F16: rounded to binary16, exact for bf16 values in
 * range), instead of their bf16 values. */
#define DFV_KV_TREE_AS_CACHE 0x100
/* Flag OR-ed into kv_format of dfv_verify_step and dfv_tree_verify_attn:
 * launch the step so that it overlaps the previous kernel of the stream
 * (programmatic dependent launch), the "pipelined" dependency mode in which
 * only the KV dependency between consecutive steps is enforced. Before that
 * kernel has completed, the step reads only q, tree_k, tree_v, parent,
 * tokens and logits -- which that kernel must not write -- and its own
 * workspace, and may OR bits into *status. ctx_len, the cache and every
 * output are read and written only after it has completed, so a chain of
 * steps over one cache gives the same results as plain launches.
 * Consecutive pipelined calls in a stream must use different workspaces
 * (two, used in turn, suffice). Needs one CTA on every SM: returns
 * DFV_ERR_UNSUPPORTED on a device with more than 256 SMs. */
#define DFV_STEP_PIPELINED 0x200

#define DFV_DTYPE_F32 0
#define DFV_DTYPE_BF16 1

#define DFV_MAX_NODES 65 /* budget <= 64 */

/* Human-readable name of a status code (static string). */
const char* dfv_status_string(dfv_status s);

/* Library version, major * 10000 + minor * 100 + patch. */
int dfv_version(void);

/* ------------------------------------------------------------------------
 * dfv_tree_verify_attn -- tree-masked attention over a Q4_0 (or F16) cache.
 *
 * Passage: "Luce DFlash: Qwen3.6-27B ..." (ai-navigate-news, ja), feature
 * list -- DDTree tree-verify (block 16, budget 22) and sliding-window flash
 * attention at decode (default window 2048) over the Q4_0 KV cache.
 *
 * out[i][h][:] = sum_k softmax_k(scale * q[i][h] . key_k) * value_k over the
 * keys visible to node i (see "Visibility" above); committed keys/values are
 * the cache's rows decoded (Q4_0 dequantised, F16 widened), tree keys/values
 * are tree_k / tree_v (with DFV_KV_TREE_AS_CACHE: those rows as the commit
 * would store them, decoded -- the reading in which tree rows are written to
 * the cache before attention and rollback truncates).
 *
 *   n_nodes        N = budget + 1, 1..DFV_MAX_NODES
 *   max_depth      bound on tree depth (block size); deeper -> DFV_DEV_DEPTH
 *   n_q_heads      Hq;  n_kv_heads Hkv; Hq % Hkv == 0, Hq <= 256
 *   head_dim       D in {64, 128, 256}
 *   window         sliding window in positions, 0 = none
 *   kv_format      DFV_KV_Q4_0 or DFV_KV_F16, optionally | DFV_KV_TREE_AS_CACHE
 *                  and | DFV_STEP_PIPELINED
 *   cache_capacity positions per head in the cache
 *   ctx_len        device int32[1], committed length C (read only)
 *   k_cache,v_cache  device cache in kv_format (layout above), read only
 *   q              device bf16 [N][Hq][D]
 *   tree_k,tree_v  device bf16 [N][Hkv][D], the tree nodes' own K/V rows
 *   parent         device int32 [N]
 *   scale          softmax scale; <= 0 means 1/sqrt(D)
 *   out            device f32 [N][Hq][D]
 *   lse            device f32 [N][Hq] (natural-log log-sum-exp), may be NULL
 *   workspace      device scratch, >= dfv_tree_verify_attn_workspace_bytes()
 *                  bytes, 256-byte aligned; zero it once before its first use
 *                  (dfv_workspace_clear); every call leaves it ready for the
 *                  next
 *   status         device uint32[1] or NULL
 *
 * Value range: |q|, |tree_k|, |tree_v| and the cache values must stay within
 * the fp16 range (the tensor-core operands are fp16).
 * ---------------------------------------------------------------------- */
size_t dfv_tree_verify_attn_workspace_bytes(int n_nodes, int n_q_heads, int n_kv_heads,
                                            int head_dim, int window, int cache_capacity);

dfv_status dfv_tree_verify_attn(int n_nodes, int max_depth, int n_q_heads, int n_kv_heads,
                                int head_dim, int window, int kv_format, int cache_capacity,
                                const int32_t* ctx_len, const void* k_cache, const void* v_cache,
                                const void* q, const void* tree_k, const void* tree_v,
                                const int32_t* parent, float scale, float* out, float* lse,
                                void* workspace, size_t workspace_bytes, uint32_t* status,
                                dfv_stream_t stream);

/* ------------------------------------------------------------------------
 * dfv_greedy_accept -- per-node argmax and greedy tree walk.
 *
 * Passage: "Luce DFlash: Qwen3.6-27B ..." (ai-navigate-news, ja), feature
 * list (greedy verification) and constraints paragraph (greedy verify only).
 *
 * argmax[i] = the lowest index of the maximum of logits[i][:] (-0.0 equals
 * +0.0; logits must hold no NaN). The walk starts at the root and, while
 * some child c of the last accepted node has tokens[c] == argmax[last],
 * accepts the lowest-index such child.
 *
 *   n_nodes       N, 1..DFV_MAX_NODES;  vocab V >= 1
 *   logits_dtype  DFV_DTYPE_F32 or DFV_DTYPE_BF16; logits device [N][V]
 *   parent        device int32 [N];  tokens device int32 [N] (draft tokens;
 *                 tokens[0] is not read)
 *   argmax        device int32 [N]                       (out)
 *   accept_len    device int32 [1], L = accepted nodes incl. root, >= 1 (out)
 *   path          device int32 [N], accepted node ids root first; entries
 *                 from L on are set to -1                (out)
 *   out_tokens    device int32 [N], tokens[path[1..L-1]] then the bonus
 *                 argmax[path[L-1]]; entries from L on are -1 (out)
 *   workspace     >= dfv_greedy_accept_workspace_bytes(); must be zeroed
 *                 once before its first use (dfv_workspace_clear); every
 *                 call leaves it zeroed again
 *   status        device uint32[1] or NULL
 * ---------------------------------------------------------------------- */
size_t dfv_greedy_accept_workspace_bytes(int n_nodes, int vocab);

dfv_status dfv_greedy_accept(int n_nodes, int vocab, int logits_dtype, const void* logits,
                             const int32_t* parent, const int32_t* tokens, int32_t* argmax,
                             int32_t* accept_len, int32_t* path, int32_t* out_tokens,
                             void* workspace, size_t workspace_bytes, uint32_t* status,
                             dfv_stream_t stream);

/* ------------------------------------------------------------------------
 * dfv_greedy_accept_static -- dfv_greedy_accept for callers that cannot
 * allocate device memory. The paper has no counterpart; this is a library
 * convenience.
 *
 * Same arguments, results and device status as dfv_greedy_accept, minus the
 * workspace: the scratch lives in a device array of
 * DFV_GREEDY_ACCEPT_STATIC_SCRATCH_BYTES bytes inside the library, which
 * every GPU that loads the library holds until the process exits. Intended
 * for code that is handed only its input and output buffers (for example a
 * plugin whose host framework owns all device memory) or that must not call
 * cudaMalloc / cudaFree because they can synchronise the device.
 *
 * - Returns DFV_ERR_WORKSPACE when the problem needs more scratch than the
 *   array holds (dfv_greedy_accept_workspace_bytes(n_nodes, vocab) >
 *   DFV_GREEDY_ACCEPT_STATIC_SCRATCH_BYTES); nothing is launched then.
 * - The first call on a device looks up the array's device address
 *   (cudaGetSymbolAddress, with that device current) and caches it; make
 *   that first call before any stream capture. The cached address is tied
 *   to the device's context: do not use the library again in a process
 *   after cudaDeviceReset.
 * - Each call clears the part of the array that must start at zero, in
 *   stream order, before its kernel. All calls on a device share the array:
 *   calls whose work overlaps on the GPU (different streams, no ordering)
 *   race and give undefined results.
 * - Allocates nothing: no cudaMalloc / cudaFree, no allocating library call.
 * ---------------------------------------------------------------------- */
#define DFV_GREEDY_ACCEPT_STATIC_SCRATCH_BYTES 16384

dfv_status dfv_greedy_accept_static(int n_nodes, int vocab, int logits_dtype, const void* logits,
                                    const int32_t* parent, const int32_t* tokens, int32_t* argmax,
                                    int32_t* accept_len, int32_t* path, int32_t* out_tokens,
                                    uint32_t* status, dfv_stream_t stream);

/* ------------------------------------------------------------------------
 * dfv_kv_commit -- commit the accepted rows, roll back the rest.
 *
 * Passage: "We got 207 tok/s with Qwen3.5-27B on an RTX 3090" (nowletus),
 * "What we ported and tuned": Q4_0 KV cache; "Luce DFlash ..." feature list:
 * tree-verify over that cache.
 *
 * For k < L = *accept_len and every KV head h, encodes tree_k[path[k]][h]
 * (and tree_v) in kv_format (DFV_KV_Q4_0: the rule below; DFV_KV_F16:
 * binary16, round-to-nearest-even) and writes it at cache position C + k,
 * C = *ctx_len;
 * then *ctx_len = C + L. Positions >= C + L are not touched (rejected nodes
 * are never written). If C + L > cache_capacity, or a path entry is outside
 * [0, n_nodes), nothing is written, *ctx_len is unchanged and a DFV_DEV_*
 * bit is set.
 *
 * Q4_0 rule per 32-value block (binary32, round-to-nearest-even, no fused
 * multiply-add): m = first element of largest magnitude, d = m / -8,
 * id = d != 0 ? 1 / d : 0, code = min(15, trunc((x * id) + 8.5)), scale
 * stored as fp16(d).
 *
 *   n_nodes       N (bounds the path entries and L)
 *   ctx_len       device int32[1], read and advanced
 *   accept_len    device int32[1];  path device int32 [>= L]
 *   tree_k/v      device bf16 [N][Hkv][D]
 *   k_cache/v_cache  device cache in kv_format, written at rows [C, C + L)
 * ---------------------------------------------------------------------- */
dfv_status dfv_kv_commit(int n_nodes, int n_kv_heads, int head_dim, int kv_format,
                         int cache_capacity, int32_t* ctx_len, const int32_t* accept_len,
                         const int32_t* path, const void* tree_k, const void* tree_v,
                         void* k_cache, void* v_cache, uint32_t* status, dfv_stream_t stream);

/* ------------------------------------------------------------------------
 * dfv_kv_quantize_rows -- fill cache rows [pos0, pos0 + n_rows) of every KV
 * head from float rows, encoded as dfv_kv_commit does (prefill).
 *
 *   src        device f32 or bf16 (src_dtype); element (row r, head h, dim
 *              c) at src[r * stride_row + h * stride_head + c] (elements)
 *   cache      device cache in kv_format (DFV_KV_Q4_0 or DFV_KV_F16),
 *              written; ctx_len is not touched
 * ---------------------------------------------------------------------- */
dfv_status dfv_kv_quantize_rows(int n_kv_heads, int head_dim, int kv_format, int cache_capacity,
                                int pos0, int n_rows, const void* src, int src_dtype,
                                int64_t stride_row, int64_t stride_head, void* cache,
                                dfv_stream_t stream);

/* ------------------------------------------------------------------------
 * dfv_verify_step -- one whole greedy tree-verify step (attention, argmax +
 * walk, commit) in ONE kernel launch on `stream`: one CTA per SM, a
 * cooperative launch (with DFV_STEP_PIPELINED: a programmatic dependent
 * launch that overlaps the previous kernel, see the flag).
 * A split of the attention waits only for the other splits of its group
 * before merging, and the walker waits only until every CTA has read the
 * committed length and reported its argmax partials. Arguments and results
 * as in the three entry points above (kv_format as for
 * dfv_tree_verify_attn: the flag changes what the attention sees, the commit
 * writes the cache format); the committed length advances by the accept
 * length. The workspace size covers either cache format.
 * `workspace` (dfv_verify_step_workspace_bytes) must be zeroed once before
 * its first use; each call leaves it ready for the next. Calls sharing a
 * workspace must not overlap on the GPU (two pipelined calls in a row would).
 * ---------------------------------------------------------------------- */
size_t dfv_verify_step_workspace_bytes(int n_nodes, int n_q_heads, int n_kv_heads, int head_dim,
                                       int window, int cache_capacity, int vocab);

dfv_status dfv_verify_step(int n_nodes, int max_depth, int n_q_heads, int n_kv_heads,
                           int head_dim, int window, int kv_format, int cache_capacity,
                           int vocab, int logits_dtype, int32_t* ctx_len, void* k_cache,
                           void* v_cache, const void* q, const void* tree_k, const void* tree_v,
                           const int32_t* parent, const int32_t* tokens, const void* logits,
                           float scale, float* out, float* lse, int32_t* argmax,
                           int32_t* accept_len, int32_t* path, int32_t* out_tokens,
                           void* workspace, size_t workspace_bytes, uint32_t* status,
                           dfv_stream_t stream);

/* Number of kernel launches one dfv_verify_step call makes for this shape
 * (host-only query; -1 for an unsupported shape). */
int dfv_verify_step_launches(int n_nodes, int n_q_heads, int n_kv_heads, int head_dim, int window,
                             int cache_capacity);

/* Zero `bytes` of a caller-owned workspace on `stream` (no allocation). */
dfv_status dfv_workspace_clear(void* workspace, size_t bytes, dfv_stream_t stream);

/* ------------------------------------------------------------------------
 * dfv_build_tree_mask -- depth and ancestor-or-self bitmask of every node
 * of a draft tree: the tree half of the visibility rule above ("Luce
 * DFlash ..." feature list: DDTree tree-verify, where a node attends to its
 * ancestors and itself). The attention computes the same values inside its
 * kernel; this helper is for callers that build their own masks.
 *
 *   n_nodes    N, 1..DFV_MAX_NODES
 *   parent     device int32 [N]; parent[0] is ignored (the root); an entry
 *              outside [0, i) is treated as 0 and sets DFV_DEV_BAD_TREE
 *   depth      device int32 [N], written: depth[0] = 0,
 *              depth[i] = depth[parent[i]] + 1
 *   anc_mask   device uint32 [N][DFV_MASK_WORDS], written: bit (t % 32) of
 *              word t / 32 of row i is set iff node t is i or an ancestor
 *              of i; bits of nodes >= N are zero
 *   status     device uint32[1] (DFV_DEV_* bits OR-ed in), may be NULL
 *
 * One launch of one CTA on `stream`. Returns DFV_ERR_INVALID for a bad
 * n_nodes or a NULL parent / depth / anc_mask, DFV_ERR_CUDA if the launch
 * fails; nothing is written then.
 * ---------------------------------------------------------------------- */
#define DFV_MASK_WORDS ((DFV_MAX_NODES + 31) / 32) /* 3 */
dfv_status dfv_build_tree_mask(int n_nodes, const int32_t* parent, int32_t* depth,
                               uint32_t* anc_mask, uint32_t* status, dfv_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* DFV_H */
