// The whole greedy tree-verify step in one launch, with the attention on the
// 5th-generation tensor cores (tcgen05, TMEM accumulators).
//
// "Luce DFlash: Qwen3.6-27B ..." (ai-navigate-news, ja), feature list: DDTree
// tree-verify (block 16, budget 22), greedy verification, Q4_0 KV cache,
// sliding-window flash attention at decode (window 2048). The step computes,
// for the N = budget + 1 tree nodes, attention over the visible committed
// keys and the node's ancestors, the argmax of every node's logits, the
// greedy walk, and the commit of the accepted rows in the cache format.
//
// One CTA per SM, one launch per step, no grid-wide barrier. CTA roles:
//   * attention units = (KV head h, 128-row tile of the head's (node, query
//     head) rows, range of 128-key chunks); the budget-22 step has 138 rows
//     per KV head, a full tile and a 10-row one. The tree chunk is processed
//     first, by the last split of each (head, tile) group;
//   * CTAs without a unit and the units of a short (<= 32-row) tile scan
//     the logits; a CTA without a unit is the walker.
// At t = 0 thread 0 reads ctx and starts 1-D bulk copies (TMA engine) of
// the unit's first K / V chunk, warp 0 those of the tile's bf16 Q rows and
// then of the CTA's logits slices, while the other warps load the tree rows.
// Then:
//   * the CTAs holding logits slices scan them into (max, lowest index)
//     partials; the walker quantises the tree rows into its smem so that the
//     commit after the walk is a plain copy;
//   * per chunk: K and V decoded ((q - 8) * d, one rounding; or binary16 rows
//     copied as they are) into 128-byte-swizzled smem; S = Q K^T by
//     tcgen05.mma into TMEM (M = 128 rows, N = 128 keys, K = D); four
//     threads per row read S from TMEM, mask (window, ancestors), exchange
//     the row max, exp2, write P (fp16) back into TMEM over S; O += P V by
//     tcgen05.mma with P from TMEM (M = 128, N = D, K = 128 keys; V as an
//     MN-major operand). The running max only moves (O rescaled in TMEM)
//     when a chunk's max exceeds it by more than 2^8, so P <= 256 fits fp16.
//     A unit with several chunks pipelines them: the next chunk's raw rows
//     are copied during the softmax, its K is decoded and its S (into a
//     second TMEM buffer) issued while P V runs, and its V decoded once P V
//     is done;
//   * each split writes its normalised O rows (fp16) with their max and sum
//     to the workspace (one bulk copy) and marks its ready word; the splits
//     of a group wait for one another (time-bounded waits) and each merges a
//     share of the group's rows by log-sum-exp;
//   * the walker waits until every other CTA has read ctx and written its
//     partials, merges the argmax partials, walks the tree in one warp,
//     copies the staged accepted rows into the cache at C..C+L-1 and
//     advances the committed length.
// A pipelined launch (programmatic dependent launch) does everything that
// reads only the step's own inputs -- the logits scan, Q, the tree -- while
// the previous kernel of the stream finishes, and waits for it before ctx.

#include <math.h>

#include "common.cuh"
#include "accept_impl.cuh"
#include "tc.cuh"

namespace dfv {

constexpr int kStepThreads = 512;   // 16 warps; four per TMEM lane quadrant
constexpr int kRowsPerTile = 128;   // UMMA M of a row tile
constexpr int kChunk = 128;         // keys per chunk (UMMA N of S, K of P V)
constexpr int kLightRows = 32;      // a tile of at most this many real rows stages logits
constexpr uint32_t kTmemCols = 512;
constexpr int kMaxStepSplits = 256;
constexpr int kMaxStepGrid = 256;   // CTAs of one launch at most
constexpr int kMaxStagedSlices = 8; // logits slices one CTA stages at most
constexpr long kSliceCostBytes = 65536;  // per-slice scan overhead (a CTA-wide reduction), in bytes of streaming
// the launch planner's cost model (see step_plan): a unit's key chunk, and
// the logits bytes a spare CTA stages and scans per microsecond
constexpr long kChunkCostNs = 6000;
constexpr long kSpareBytesPerUs = 32000;
constexpr float kRescaleLog2 = 8.0f;
constexpr int kLogitVecs = 16;      // 16-byte logits vectors a thread keeps in flight

struct StepPlan {
  int rows, n_grp, splits, units, grid, lunits, lchunks, lchunk_len, lbulk, lstride, lper, smem;
  int walker, walker_local;
  uint32_t lslot[kMaxStepGrid];   // per CTA: first logits slice | count << 16
  size_t ws_bar, ws_arg, ws_qrows, ws_ml, ws_o, ws_total;
};

struct StepParams {
  int n_nodes, max_depth, hq, hkv, group, window, capacity, vocab, logits_dtype;
  int rows;          // N * group: (node, query head) rows of one KV head
  int n_grp;         // 128-row tiles per KV head
  int splits, units, lunits, lchunks, lchunk_len, lbulk;
  int lstride;       // bytes between staged slices
  int lper;          // staged slices per half of the staging area (one round)
  uint32_t group_m;  // ceil(2^32 / group) (0 when group == 1): row -> node by multiply-high
  int do_accept;
  int tree_q;        // attend Q4_0-quantised-and-dequantised tree rows
  int pipelined;     // launched to overlap the previous kernel of the stream
  int walker;        // CTA that merges the argmax partials, walks and commits
  int walker_local;  // 1: it quantises the tree rows into its own smem
  float scale_log2;
  int32_t* ctx_len;
  uint8_t* k_cache;
  uint8_t* v_cache;
  const __nv_bfloat16* q;
  const __nv_bfloat16* tree_k;
  const __nv_bfloat16* tree_v;
  const int32_t* parent;
  const int32_t* tokens;
  const void* logits;
  float* out;
  float* lse;
  int32_t* argmax;
  int32_t* accept_len;
  int32_t* path;
  int32_t* out_tokens;
  unsigned int* bar;        // [2] CTAs done with ctx and their argmax partials
                            // (the walker waits for exactly grid - 1 reports,
                            // then resets it); [4 + 2 g]: arrivals (low 16
                            // bits) and generation of split group g
  unsigned int* ready;      // [units] generation + 1 once the unit's partial is written
  ArgPartial* arg_part;     // [lunits]
  uint8_t* qrows;           // [N][Hkv][2][row bytes]
  uint8_t* part;            // [units][128] rows of kPartRowBytes: O / sum (fp16),
                            // then (running max, log2 units; sum)
  uint32_t* status;
  uint32_t lslot[kMaxStepGrid];   // per CTA: first staged logits slice | count << 16
};

// One row of a split's partial: D fp16 values, the row's (max, sum), 8
// bytes of padding (rows stay 16-byte aligned; consecutive rows of a staged
// tile fall on different banks).
template <int D>
constexpr int kPartRowBytes = D * 2 + 16;

// Dynamic shared memory map (bytes from a 1024-aligned base).
template <int D>
struct StepSmem {
  static constexpr int kRowB = D / 32 * 18;
  static constexpr bool kBulk = (kRowB % 16) == 0;
  static constexpr int kTileB = kRowsPerTile * D * 2;        // one [128][D] fp16 tile
  static constexpr int kQ = 0;                               // Q of the tile
  static constexpr int kK = kQ + kTileB;                     // K^
  static constexpr int kKBytes0 = kChunk * D * 2;
  static constexpr int kKBytes1 = kChunk * kChunk * 2;
  static constexpr int kKBytes = kKBytes0 > kKBytes1 ? kKBytes0 : kKBytes1;
  static constexpr int kV = kK + kKBytes;                    // V^; raw K, raw V land at its end first
  static constexpr int kRawK = kChunk * D * 2 - 2 * kChunk * kRowB;   // raw K's offset in sV
  static constexpr int kRawV = kRawK + kChunk * kRowB;                // raw V's offset in sV
  static constexpr int kQStage = kK;                         // bf16 Q rows land here (sK, then sV)
  // raw K / V of a unit's later chunks, copied while the chunk before is
  // still in its softmax and P V: raw K in sK (free once S of that chunk is
  // done; P is in TMEM), raw V in a region of its own
  static constexpr int kRawK2 = kKBytes1;                    // offset in sK
  static constexpr int kRawV2 = kV + kChunk * D * 2;
  static constexpr int kBars = kRawV2 + (kBulk ? kChunk * kRowB : 0);
  static constexpr int kSpareStageBytes = kBars;             // logits staging of a CTA without a unit
  // logits staging of a unit whose tile has at most kLightRows real rows:
  // past its staged Q rows, up to the raw K / V (free until the dequant)
  static constexpr int kUnitStage = kK + kLightRows * D * 2;
  static constexpr int kUnitStageBytes = kV + kRawK - kUnitStage;
  static constexpr int kBytes = kBars + 64 + 1024;           // + alignment slack
  static_assert(2 * kChunk * kRowB <= kChunk * D * 2, "raw K and V fit in sV");
  static_assert(kRawK % 16 == 0 && kRawV % 16 == 0, "bulk-copy destinations 16-byte aligned");
  static_assert(kRowsPerTile * D * 2 <= kKBytes + kRawK, "staged Q rows stay clear of raw K / V");
  static_assert(kRowsPerTile * (D * 2 + 16) <= kV, "epilogue staging fits in sQ + sK");
  static_assert(!kBulk || kRawK2 + kChunk * kRowB <= kKBytes, "next raw K fits in sK");
  static_assert(kRawK2 % 16 == 0 && kRawV2 % 16 == 0, "bulk-copy destinations 16-byte aligned");
};

// ---------------------------------------------------------------- small helpers

__device__ __forceinline__ uint4 bf16x8_to_f16x8(uint4 v) {
  const __nv_bfloat162* b = reinterpret_cast<const __nv_bfloat162*>(&v);
  uint4 o;
  uint32_t* ov = reinterpret_cast<uint32_t*>(&o);
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const float2 f = __bfloat1622float2(b[e]);
    ov[e] = pack_half2(f.x, f.y);
  }
  return o;
}

// One Q4_0 block -> 32 fp16 values in four 16-byte chunks (chunk 0 =
// values 0..7, 1 = 8..15: the low nibbles of code bytes 0..15; 2 = 16..23,
// 3 = 24..31: their high nibbles). `code` holds the 16 code bytes as four
// little-endian words, `dbits` the fp16 scale. Each code word becomes four
// half2 of exact integers 1024 + q (the nibble under the exponent of 1024),
// then (x - 1032) * d rounds once to fp16.
__device__ __forceinline__ void q4_0_block_chunks(const uint32_t* code, uint32_t dbits, uint4* out) {
  const __half dh = __ushort_as_half(static_cast<unsigned short>(dbits & 0xFFFFu));
  const __half2 d2 = __halves2half2(dh, dh);
  const __half2 bias = __float2half2_rn(1032.0f);
  uint32_t* o = reinterpret_cast<uint32_t*>(out);
  auto scale = [&](uint32_t x) {
    const __half2 v = __hmul2(__hsub2(*reinterpret_cast<const __half2*>(&x), bias), d2);
    return *reinterpret_cast<const uint32_t*>(&v);
  };
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const uint32_t a = __byte_perm(code[k], 0u, 0x4140);   // [b0, 0, b1, 0]
    const uint32_t b = __byte_perm(code[k], 0u, 0x4342);   // [b2, 0, b3, 0]
    const int cl = k >> 1, pos = (k & 1) * 2;
    o[cl * 4 + pos] = scale((a & 0x000F000Fu) | 0x64006400u);                // values 4k, 4k+1
    o[cl * 4 + pos + 1] = scale((b & 0x000F000Fu) | 0x64006400u);            // 4k+2, 4k+3
    o[(2 + cl) * 4 + pos] = scale(((a >> 4) & 0x000F000Fu) | 0x64006400u);   // 16+4k, ...
    o[(2 + cl) * 4 + pos + 1] = scale(((b >> 4) & 0x000F000Fu) | 0x64006400u);
  }
}

// Two consecutive Q4_0 blocks (36 bytes as nine little-endian words) -> 64
// fp16 values in eight 16-byte chunks. The first block's code bytes start
// two bytes into the words, so they are realigned by funnel shifts.
__device__ __forceinline__ void q4_0_pair_chunks(const uint32_t* w, uint4* out) {
  uint32_t ca[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) ca[i] = __funnelshift_r(w[i], w[i + 1], 16);
  q4_0_block_chunks(ca, w[0], out);
  q4_0_block_chunks(w + 5, w[4] >> 16, out + 4);
}

__device__ __forceinline__ uint32_t ld_acquire_gpu(const unsigned int* a) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(a) : "memory");
  return v;
}

// Waits (time-bounded) until ready[0..n) all hold `tag`; one warp polls,
// lane i the words i, i + 32, ...; false on timeout.
__device__ __forceinline__ bool wait_ready(const unsigned int* ready, int n, uint32_t tag) {
  const int lane = threadIdx.x & 31;
  bool ok = true;
  for (int i = lane; i < n && ok; i += 32)
    ok = wait_bounded([&]() { return ld_acquire_gpu(ready + i) == tag; });
  return __all_sync(0xffffffffu, ok);
}

// n / d for n < 2^16 and 2 <= d <= 256 as the high word of n * ceil(2^32 / d)
// (exact in that range); m == 0 stands for d == 1.
__device__ __forceinline__ int div_small(int n, uint32_t m) {
  return m == 0u ? n : static_cast<int>(__umulhi(static_cast<uint32_t>(n), m));
}

// Maximum of a float over the CTA, returned to every thread.
__device__ __forceinline__ float block_max(float v) {
  __shared__ float sm[kStepThreads / 32];
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  if ((threadIdx.x & 31) == 0) sm[threadIdx.x >> 5] = v;
  __syncthreads();
  float m = sm[0];
#pragma unroll
  for (int w = 1; w < kStepThreads / 32; ++w) m = fmaxf(m, sm[w]);
  __syncthreads();
  return m;
}

// Thread 0 waits for an mbarrier phase; the CTA learns the outcome.
__device__ __forceinline__ bool cta_wait(uint64_t* bar, uint32_t parity, int* s_flag,
                                         uint32_t* status) {
  if (threadIdx.x == 0) {
    const bool ok = mbar_wait_bounded(bar, parity);
    if (!ok) report(status, DFV_DEV_TIMEOUT);
    *s_flag = ok ? 1 : 0;
  }
  __syncthreads();
  return *s_flag != 0;
}

// ---------------------------------------------------------------- the kernel

// Thread 0: the bulk copies of round r of this CTA's staged logits slices
// [ls0, ls0 + lsn): slices r * lper .. into half (r & 1) of the staging
// area, completing on bars[r & 1].
template <typename LT>
__device__ __forceinline__ void issue_slices(const StepParams& p, uint8_t* lstage, int ls0, int lsn, int r,
                                             uint64_t* bars) {
  constexpr int esz = static_cast<int>(sizeof(LT));
  const int k0 = r * p.lper, k1 = min(lsn, k0 + p.lper);
  uint8_t* buf = lstage + (r & 1) * p.lper * p.lstride;
  uint32_t total = 0;
  for (int k = k0; k < k1; ++k) {
    const int ch = (ls0 + k) % p.lchunks;
    const int b0 = ch * p.lchunk_len, b1 = max(b0, min(p.vocab, b0 + p.lchunk_len));
    total += static_cast<uint32_t>((b1 - b0) * esz);
  }
  fence_proxy_async_smem();   // the buffer was last read through the generic proxy
  mbar_arrive_expect_tx(bars + (r & 1), total);
  for (int k = k0; k < k1; ++k) {
    const int u = ls0 + k, node = u / p.lchunks, ch = u % p.lchunks;
    const int b0 = ch * p.lchunk_len, b1 = max(b0, min(p.vocab, b0 + p.lchunk_len));
    if (b1 > b0)
      bulk_g2s(buf + (k - k0) * p.lstride,
               static_cast<const uint8_t*>(p.logits) + (static_cast<size_t>(node) * p.vocab + b0) * esz,
               static_cast<uint32_t>((b1 - b0) * esz), bars + (r & 1));
  }
}

// Argmax partials of this CTA's staged logits slices [ls0, ls0 + lsn),
// round by round: rounds 0 and 1 were issued at entry into the two halves
// of the staging area, round r + 2 is issued into the half round r frees.
// One pass per slice: four independent chains per thread, each keeping its
// running maximum and the first vector that reached it; then the lowest
// vector holding the thread's maximum is re-read for the lowest element
// index, and the (max, lowest index) pairs merge across the CTA.
template <typename LT>
__device__ __forceinline__ void scan_slices(const StepParams& p, uint8_t* lstage, int ls0, int lsn,
                                         uint64_t* bars, int* s_ok) {
  constexpr int esz = static_cast<int>(sizeof(LT));
  const int tid = threadIdx.x;
  const int rounds = (lsn + p.lper - 1) / p.lper;
#pragma unroll 1
  for (int rd = 0; rd < rounds; ++rd) {
  const bool ok = cta_wait(bars + (rd & 1), (rd >> 1) & 1, s_ok, p.status);
  const int k0 = rd * p.lper, k1 = min(lsn, k0 + p.lper);
#pragma unroll 1
  for (int k = k0; k < k1; ++k) {
    const int u = ls0 + k;
    const int lbegin = (u % p.lchunks) * p.lchunk_len;
    const int lend = max(lbegin, min(p.vocab, lbegin + p.lchunk_len));
    const int lnvec = (lend - lbegin) * esz / 16;
    const uint4* sv = reinterpret_cast<const uint4*>(lstage + (rd & 1) * p.lper * p.lstride +
                                                     (k - k0) * p.lstride);
    float best = -INFINITY;
    int bidx = INT_MAX;
    if (ok) {
      float bk[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
      int vk[4] = {INT_MAX, INT_MAX, INT_MAX, INT_MAX};
#pragma unroll 1
      for (int v0 = tid; v0 < lnvec; v0 += 4 * kStepThreads) {
        uint4 x[4];
#pragma unroll
        for (int c = 0; c < 4; ++c)
          if (v0 + c * kStepThreads < lnvec) x[c] = sv[v0 + c * kStepThreads];
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          if (v0 + c * kStepThreads < lnvec) {
            float mf;
            if constexpr (esz == 2) {
              const __nv_bfloat162* b = reinterpret_cast<const __nv_bfloat162*>(&x[c]);
              const __nv_bfloat162 m = __hmax2(__hmax2(b[0], b[1]), __hmax2(b[2], b[3]));
              mf = fmaxf(__low2float(m), __high2float(m));
            } else {
              const float* f = reinterpret_cast<const float*>(&x[c]);
              mf = fmaxf(fmaxf(f[0], f[1]), fmaxf(f[2], f[3]));
            }
            // the first vector is taken even at -inf (a slice of -inf still
            // has an argmax: its first element)
            if (mf > bk[c] || (vk[c] == INT_MAX && mf == mf)) { bk[c] = mf; vk[c] = v0 + c * kStepThreads; }
          }
        }
      }
      best = fmaxf(fmaxf(bk[0], bk[1]), fmaxf(bk[2], bk[3]));
      int vm = INT_MAX;
#pragma unroll
      for (int c = 0; c < 4; ++c)
        if (bk[c] == best && vk[c] < vm) vm = vk[c];
      if (vm != INT_MAX) {
        const uint4 x = sv[vm];
        if constexpr (esz == 2) {
          const __nv_bfloat16* be = reinterpret_cast<const __nv_bfloat16*>(&x);
#pragma unroll
          for (int e = 7; e >= 0; --e)
            if (__bfloat162float(be[e]) == best) bidx = lbegin + vm * 8 + e;
        } else {
          const float* f = reinterpret_cast<const float*>(&x);
#pragma unroll
          for (int e = 3; e >= 0; --e)
            if (f[e] == best) bidx = lbegin + vm * 4 + e;
        }
      }
      if (bidx == INT_MAX) best = -INFINITY;   // no element: loses every merge
    }
    block_argmax<kStepThreads>(best, bidx);
    if (tid == 0) {
      p.arg_part[u].v = best;
      p.arg_part[u].idx = bidx;
    }
    __syncthreads();   // the staging buffer is free again
  }
  if (tid == 0 && rd + 2 < rounds) issue_slices<LT>(p, lstage, ls0, lsn, rd + 2, bars);
  }
}

// Argmax partials of logits slices blk, blk + G, ... by plain loads (when the
// slices cannot be staged in smem).
template <typename LT>
__device__ __forceinline__ void plain_slices(const StepParams& p, int blk, int G) {
  for (int u = blk; u < p.lunits; u += G) {
    const int node = u / p.lchunks, ch = u % p.lchunks;
    const int begin = ch * p.lchunk_len;
    const int end = min(p.vocab, begin + p.lchunk_len);
    float best = -INFINITY;
    int bidx = INT_MAX;
    chunk_argmax<LT, 8, kStepThreads>(static_cast<const LT*>(p.logits) + static_cast<size_t>(node) * p.vocab,
                                      begin, end, best, bidx);
    block_argmax<kStepThreads>(best, bidx);
    if (threadIdx.x == 0) {
      p.arg_part[u].v = best;
      p.arg_part[u].idx = bidx;
    }
    __syncthreads();
  }
}

// Q4_0 blocks [b0, b1) of the tree's key / value rows, laid out
// [node][Hkv][K, V][row bytes] at qdst.
template <int D, int FMT>
__device__ __forceinline__ void prequant_tree(const StepParams& p, uint8_t* qdst, int b0, int b1) {
  constexpr int NB = D / 32;
  constexpr int kRowB = kv_row_bytes(FMT, D);
  if constexpr (FMT == DFV_KV_F16) {
    // items of eight values: bf16 -> binary16 (nearest even); b0, b1 count
    // 32-value blocks, four items each
    for (int it = 4 * b0 + static_cast<int>(threadIdx.x); it < 4 * b1; it += kStepThreads) {
      const int c = it % (D / 8);
      const int kv = (it / (D / 8)) & 1;
      const int hh = (it / (2 * (D / 8))) % p.hkv;
      const int t = it / (2 * (D / 8) * p.hkv);
      const uint4 v = *reinterpret_cast<const uint4*>(
          (kv ? p.tree_v : p.tree_k) + (static_cast<size_t>(t) * p.hkv + hh) * D + c * 8);
      *reinterpret_cast<uint4*>(qdst + ((static_cast<size_t>(t) * p.hkv + hh) * 2 + kv) * kRowB + c * 16) =
          bf16x8_to_f16x8_rn(v);
    }
  } else {
  for (int it = b0 + static_cast<int>(threadIdx.x); it < b1; it += kStepThreads) {
    const int b = it % NB;
    const int kv = (it / NB) & 1;
    const int hh = (it / (2 * NB)) % p.hkv;
    const int t = it / (2 * NB * p.hkv);
    const uint4* v = reinterpret_cast<const uint4*>(
        (kv ? p.tree_v : p.tree_k) + (static_cast<size_t>(t) * p.hkv + hh) * D + b * 32);
    uint4 r4[4];
#pragma unroll
    for (int u4 = 0; u4 < 4; ++u4) r4[u4] = v[u4];
    float x[32];
#pragma unroll
    for (int u4 = 0; u4 < 4; ++u4) {
      const __nv_bfloat162* hb = reinterpret_cast<const __nv_bfloat162*>(&r4[u4]);
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float2 f = __bfloat1622float2(hb[e]);
        x[u4 * 8 + 2 * e] = f.x;
        x[u4 * 8 + 2 * e + 1] = f.y;
      }
    }
    q4_0_quantize_block(x, qdst + ((static_cast<size_t>(t) * p.hkv + hh) * 2 + kv) * kRowB + b * 18);
  }
  }
}

// The walker: waits until every other CTA has read ctx and written what it
// owes (argmax partials, tree rows), merges the argmax partials per node,
// walks the tree from the root and commits the accepted rows to the cache.
template <int D, int FMT>
__device__ __forceinline__ void walker_tail(const StepParams& p, int G, int C, bool ctx_ok, uint8_t* sQ,
                                         const uint8_t* sK, const int* s_wpar, const int* s_wtok) {
  using L = StepSmem<D>;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int N = p.n_nodes;
  __shared__ int s_ok;
  if (tid == 0) {
    // exactly G - 1 reports (one per other CTA); a count that never equals
    // it (a corrupted workspace) ends in a timeout, and nothing is committed
    volatile unsigned int* done = p.bar + 2;
    const unsigned int want = static_cast<unsigned int>(G - 1);
    const bool ok = wait_bounded([&]() {
      if (*done == want) return true;
      __nanosleep(32);
      return false;
    });
    __threadfence();
    *done = 0u;                        // ready for the next launch
    p.bar[3] = 0u;                     // the units' "copies issued" count too
    if (!ok) report(p.status, DFV_DEV_TIMEOUT);
    s_ok = ok ? 1 : 0;
  }
  __syncthreads();
  if (!s_ok) return;
  __shared__ int s_am[kMaxNodes];
  __shared__ int s_path[kMaxNodes];
  __shared__ int s_L;
  // every partial in one round of loads (staged in sQ), then per node
  ArgPartial* s_ap = reinterpret_cast<ArgPartial*>(sQ);
  for (int i = tid; i < p.lunits; i += kStepThreads) {
    ArgPartial a;
    a.v = __ldcg(&p.arg_part[i].v);
    a.idx = __ldcg(&p.arg_part[i].idx);
    s_ap[i] = a;
  }
  __syncthreads();
  for (int node = warp; node < N; node += kStepThreads / 32) {
    float best = -INFINITY;
    int bidx = INT_MAX;
    for (int c = lane; c < p.lchunks; c += 32) {
      const ArgPartial a = s_ap[node * p.lchunks + c];
      if (beats(a.v, a.idx, best, bidx)) { best = a.v; bidx = a.idx; }
    }
    warp_argmax(best, bidx);
    if (lane == 0) {
      s_am[node] = bidx;
      p.argmax[node] = bidx;
    }
  }
  __syncthreads();
  if (warp == 0) {
    int par[3], tok[3];
#pragma unroll
    for (int s = 0; s < 3; ++s) {
      const int n = lane + 32 * s;
      par[s] = -2;
      tok[s] = 0;
      if (n >= 1 && n < N) {
        int pa = s_wpar[n];
        if (pa < 0 || pa >= n) pa = 0;
        par[s] = pa;
        tok[s] = s_wtok[n];
      }
    }
    int cur = 0, Lw = 1;
    if (lane == 0) s_path[0] = 0;
    for (int itw = 0; itw < N; ++itw) {
      const int t = s_am[cur];
      const unsigned b0 = __ballot_sync(0xffffffffu, par[0] == cur && tok[0] == t);
      const unsigned b1 = __ballot_sync(0xffffffffu, par[1] == cur && tok[1] == t);
      const unsigned b2 = __ballot_sync(0xffffffffu, par[2] == cur && tok[2] == t);
      int next = -1;
      if (b0) next = __ffs(b0) - 1;
      else if (b1) next = 31 + __ffs(b1);
      else if (b2) next = 63 + __ffs(b2);
      if (next < 0) break;
      if (lane == 0) s_path[Lw] = next;
      ++Lw;
      cur = next;
    }
    __syncwarp();
    for (int k = lane; k < N; k += 32) {
      p.path[k] = k < Lw ? s_path[k] : -1;
      int ot = -1;
      if (k < Lw - 1) ot = s_wtok[s_path[k + 1]];
      else if (k == Lw - 1) ot = s_am[s_path[Lw - 1]];
      p.out_tokens[k] = ot;
    }
    if (lane == 0) {
      *p.accept_len = Lw;
      s_L = Lw;
    }
  }
  __syncthreads();
  const int Lc = s_L, Cc = C;
  if (!ctx_ok) {
    // the committed length was outside [0, capacity] (reported at entry):
    // nothing is committed
  } else if (Cc + Lc > p.capacity) {
    if (tid == 0) report(p.status, DFV_DEV_CAPACITY);
  } else {
    constexpr int kCRowB = kv_row_bytes(FMT, D);   // bytes of one cache row
    constexpr int W4 = kCRowB / 4;
    const int total = Lc * p.hkv * 2 * W4;
    for (int it = tid; it < total; it += kStepThreads) {
      const int w = it % W4;
      const int kv = (it / W4) & 1;
      const int hh = (it / (2 * W4)) % p.hkv;
      const int k = it / (2 * W4 * p.hkv);
      const size_t so = ((static_cast<size_t>(s_path[k]) * p.hkv + hh) * 2 + kv) * kCRowB;
      uint32_t* dst = reinterpret_cast<uint32_t*>(
          (kv ? p.v_cache : p.k_cache) + (static_cast<size_t>(hh) * p.capacity + Cc + k) * kCRowB);
      dst[w] = p.walker_local ? reinterpret_cast<const uint32_t*>(sK + so)[w]
                              : __ldcg(reinterpret_cast<const uint32_t*>(p.qrows + so) + w);
    }
    __syncthreads();
    if (tid == 0) *p.ctx_len = Cc + Lc;
  }
}

template <int D, typename LT, int FMT>
__global__ void __launch_bounds__(kStepThreads, 1) step_kernel(const __grid_constant__ StepParams p) {
  using L = StepSmem<D>;
  constexpr bool kQ4 = FMT == DFV_KV_Q4_0;   // else binary16 cache rows
  constexpr int NB = D / 32;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  // swizzle atoms need 1024-byte aligned bases; the launch adds 1 KB of slack
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint8_t* sQ = smem + L::kQ;
  uint8_t* sK = smem + L::kK;
  uint8_t* sV = smem + L::kV;
  uint64_t* bar_kv = reinterpret_cast<uint64_t*>(smem + L::kBars);
  uint64_t* bar_mma = bar_kv + 1;
  uint64_t* bar_lg = bar_kv + 2;     // bar_lg[0..1]: the two halves of the logits staging
  uint64_t* bar_lg2 = bar_kv + 3;
  uint64_t* bar_q = bar_kv + 4;
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(bar_kv + 5);
  uint64_t* bar_s = bar_kv + 6;      // S of a chunk done

  __shared__ int s_J[kMaxNodes], s_dep[kMaxNodes];
  __shared__ uint32_t s_anc[kMaxNodes][kMaskWords];
  __shared__ int s_row_node[kRowsPerTile], s_row_lo[kRowsPerTile];
  __shared__ float s_pmax[4][kRowsPerTile];
  __shared__ float s_l[4][kRowsPerTile];
  __shared__ int s_ok;
  __shared__ int s_wpar[kMaxNodes], s_wtok[kMaxNodes];

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int G = gridDim.x;
  // A pipelined step hands the roles out in reverse, so that the CTAs that
  // start first, on the SMs the previous step frees first, are the walker
  // and the logits CTAs: their work does not wait for that step.
  const int blk = p.pipelined ? G - 1 - static_cast<int>(blockIdx.x) : static_cast<int>(blockIdx.x);
  const int N = p.n_nodes;
  grid_dep_launch_dependents();   // the next step may start on SMs this one frees

  // ---- this CTA's attention unit
  const int unit = blk < p.units ? blk : -1;
  int h = 0, grp = 0, split = 0;
  if (unit >= 0) {
    split = unit % p.splits;
    grp = (unit / p.splits) % p.n_grp;
    h = unit / (p.splits * p.n_grp);
  }
  // the context length, read once by thread 0 (with acquire semantics, so
  // that its report to the walker below cannot overtake it) and shared
  // through smem after the first barrier
  __shared__ int s_C;
  __shared__ int s_ctx_ok;     // ctx was inside [0, capacity]
  __shared__ uint32_t s_tag;   // this launch's ready tag of the unit's group
  // Chunks [c0, c1) of the unit; the tree chunk (N <= 65 keys: one chunk,
  // the last, held by the last split) is processed first, then the
  // committed ones. first_kv: the first chunk processed is committed.
  int C = 0, lo_min = 0, n_cc = 0, T = 0, c0 = 0, c1 = 0, n_tree = 0;
  bool first_kv = false;
  auto derive = [&]() {
    lo_min = p.window > 0 ? max(0, C - p.window + 1) : 0;
    n_cc = (C - lo_min + kChunk - 1) / kChunk;                 // committed chunks
    T = n_cc + 1;                                              // + the tree chunk
    if (unit >= 0) {
      // floor(s * T / splits) without a 64-bit product: T = q * splits + r
      const int q = T / p.splits, r = T - q * p.splits;
      c0 = split * q + split * r / p.splits;
      c1 = (split + 1) * q + (split + 1) * r / p.splits;
      n_tree = c1 > n_cc ? 1 : 0;
      first_kv = n_tree == 0 && c0 < c1;
    }
  };

  // raw K / V of chunk cc -> dk / dv (read into registers before K^ / V^
  // are written over them); thread 0 counts the copies not yet waited for
  int kv_pending = 0;
  auto issue_kv = [&](int cc, uint8_t* dk, uint8_t* dv) {
    const int j0 = lo_min + cc * kChunk;
    const int nk = min(kChunk, C - j0);
    const uint32_t bytes = static_cast<uint32_t>(nk * L::kRowB);
    const size_t off = (static_cast<size_t>(h) * p.capacity + j0) * L::kRowB;
    fence_proxy_async_smem();
    mbar_arrive_expect_tx(bar_kv, 2 * bytes);
    bulk_g2s(dk, p.k_cache + off, bytes, bar_kv);
    bulk_g2s(dv, p.v_cache + off, bytes, bar_kv);
    ++kv_pending;
  };
  // the tile's rows [128 grp, 128 grp + rows_g): node n's query heads of KV
  // head h are contiguous, so one bulk copy per node lands the bf16 rows in
  // order at sK (then on into sV, clear of the raw K / V)
  const int rows_g = unit >= 0 ? min(kRowsPerTile, p.rows - grp * kRowsPerTile) : 0;
  auto issue_q = [&]() {   // by the 32 lanes of warp 0, node n0 + lane + 32 k each
    const int start = grp * kRowsPerTile, end = start + rows_g;
    for (int n = div_small(start, p.group_m) + lane; n * p.group < end; n += 32) {
      const int j0 = max(start, n * p.group) - n * p.group, j1 = min(end, (n + 1) * p.group) - n * p.group;
      bulk_g2s(smem + L::kQStage + static_cast<size_t>(n * p.group + j0 - start) * D * 2,
               p.q + (static_cast<size_t>(n) * p.hq + h * p.group + j0) * D,
               static_cast<uint32_t>((j1 - j0) * D * 2), bar_q);
    }
  };

  // The logits slices [ls0, ls0 + lsn) of a CTA without a unit land in smem
  // by TMA at t = 0 (slice k at sQ + k * lstride) and are scanned as soon as
  // they have landed. When the slices cannot be staged, every CTA takes
  // slices blk, blk + G, ... with plain loads instead.
  const uint32_t le = p.do_accept && p.lbulk ? p.lslot[blk] : 0u;
  const int ls0 = static_cast<int>(le & 0xFFFFu), lsn = static_cast<int>(le >> 16);
  const bool lreg = lsn > 0;
  uint8_t* lstage = unit >= 0 ? smem + L::kUnitStage : sQ;
  // A CTA reports to the walker ("ctx read, my writes done") once everything
  // the walker reads from it is written: its argmax partials, its share of
  // the quantised tree rows when those go through the workspace. A CTA with
  // neither reports right after reading ctx.
  const bool qshare = p.do_accept && !p.walker_local;
  const bool has_slices = lreg || (p.do_accept && !p.lbulk && blk < p.lunits);
  const bool late_signal = has_slices || qshare;
  // the late report: after a barrier that follows every write of the CTA
  auto signal_done = [&]() {
    if (p.do_accept && blk != p.walker && tid == 0) {
      __threadfence();
      atomicAdd(p.bar + 2, 1u);
    }
  };

  // ================================================================ phase A
  unsigned int arrive_old = 0;   // thread 0: its add to the split group's word
  // Thread 0: the read of ctx, the split group's arrival and the first K / V
  // copy. Everything a step reads or writes that the previous step may
  // write (ctx, the cache, the outputs) comes after this.
  auto ctx_and_first_kv = [&]() {
    C = static_cast<int>(ld_acquire_gpu(reinterpret_cast<const unsigned int*>(p.ctx_len)));
    // the group arrival's old value is only needed at the end of the unit
    if (unit >= 0 && p.splits > 1) arrive_old = atomicAdd(p.bar + 4 + 2 * (unit / p.splits), 1u);
    s_ctx_ok = 1;
    if (C < 0 || C > p.capacity) {
      if (blk == 0) report(p.status, DFV_DEV_CTX);
      C = C < 0 ? 0 : p.capacity;
      s_ctx_ok = 0;
    }
    s_C = C;
    derive();
    if constexpr (L::kBulk && kQ4) {
      if (first_kv) issue_kv(c0, sV + L::kRawK, sV + L::kRawV);
    }
  };
  // Warp 0 first, before any load of its own (the barrier-init fence would
  // wait for them). Thread 0: the barriers; the read of ctx and the first K /
  // V copy (not yet when pipelined); then warp 0's lanes issue the Q rows'
  // copies, and, on a CTA without a unit, thread 0 the logits copies. Those
  // wait (non-pipelined) until every unit has issued its K / V and Q copies,
  // so that the attention's bytes are ahead of the logits in the memory
  // system; the walker resets the count. Meanwhile warps 1..15 load the tree
  // rows, allocate TMEM and build the tree masks; a CTA-wide barrier then
  // makes the barriers and ctx visible to all.
  if (warp == 0) {
    if (tid == 0) {
      mbar_init(bar_kv, 1);
      mbar_init(bar_mma, 1);
      mbar_init(bar_lg, 1);
      mbar_init(bar_q, 1);
      mbar_init(bar_s, 1);
      mbar_init(bar_lg2, 1);
      fence_mbar_init();
      if (!p.pipelined) ctx_and_first_kv();
      if (unit >= 0) mbar_arrive_expect_tx(bar_q, static_cast<uint32_t>(rows_g * D * 2));
    }
    __syncwarp();
    if (unit >= 0) issue_q();
    __syncwarp();
    if (tid == 0) {
      if (unit >= 0 && !p.pipelined && p.do_accept) atomicAdd(p.bar + 3, 1u);
      if (lreg) {
        if (!p.pipelined && unit < 0) {
          volatile unsigned int* issued = p.bar + 3;
          const unsigned int want = static_cast<unsigned int>(p.units);
          wait_bounded([&]() {
            if (*issued >= want) return true;
            __nanosleep(64);
            return false;
          });   // ordering only: the copies below go ahead either way
        }
        issue_slices<LT>(p, lstage, ls0, lsn, 0, bar_lg);
        if (lsn > p.lper) issue_slices<LT>(p, lstage, ls0, lsn, 1, bar_lg);
      }
      // nothing for the walker to wait for but the read of ctx above
      if (!p.pipelined && p.do_accept && blk != p.walker && !late_signal) atomicAdd(p.bar + 2, 1u);
    }
  }
  // Warps 1..15: the last split's tree rows (its first chunk; this thread's
  // first TP 16-byte pieces, converted when the chunk is built).
  constexpr int kLoaders = kStepThreads - 32;
  const int li = tid - 32;                       // loader index (< 0: warp 0)
  constexpr int TP = 4;
  const bool tree_split = unit >= 0 && split == p.splits - 1;
  const int nt_all = min(kChunk, N);
  const int tree_real = 2 * nt_all * (D / 8);     // 16-byte pieces with data
  uint4 tv[TP];
#pragma unroll
  for (int u = 0; u < TP; ++u) {
    const int it = li + u * kLoaders;
    tv[u] = make_uint4(0u, 0u, 0u, 0u);
    if (li >= 0 && tree_split && it < tree_real) {
      const int ka = it / (D / 8), c = it % (D / 8);
      const int kvi = ka >= nt_all ? 1 : 0, key = ka - kvi * nt_all;
      tv[u] = __ldg(reinterpret_cast<const uint4*>(
          (kvi ? p.tree_v : p.tree_k) + (static_cast<size_t>(key) * p.hkv + h) * D + c * 8));
    }
  }
  if (unit >= 0 && warp == 2) {
    tc::tmem_alloc(s_tmem, kTmemCols);
    tc::fence_before_sync();
  }
  // ---- tree: depth and ancestor-or-self masks, by pointer jumping in one
  // warp while the copies are in flight; ceil(log2 N) rounds cover every
  // depth (< N)
  if (unit >= 0 && warp == 1) {
#pragma unroll
    for (int k = 0; k < 3; ++k) {
      const int n = lane + 32 * k;
      if (n < N) {
        int pa = n == 0 ? -1 : p.parent[n];
        if (n > 0 && (pa < 0 || pa >= n)) {
          if (blk == 0) report(p.status, DFV_DEV_BAD_TREE);
          pa = 0;
        }
        s_J[n] = pa;
        s_dep[n] = n > 0 ? 1 : 0;
#pragma unroll
        for (int w = 0; w < kMaskWords; ++w) s_anc[n][w] = (n >> 5) == w ? (1u << (n & 31)) : 0u;
      }
    }
    int rounds = 0;
    while ((1 << rounds) < N) ++rounds;
    __syncwarp();
#pragma unroll 1
    for (int round = 0; round < rounds; ++round) {
      int jj[3], nd[3], nj[3];
      uint32_t nm[3][kMaskWords];
#pragma unroll
      for (int k = 0; k < 3; ++k) {
        const int n = lane + 32 * k;
        jj[k] = -1;
        if (n < N) {
          jj[k] = s_J[n];
          if (jj[k] >= 0) {
            nd[k] = s_dep[n] + s_dep[jj[k]];
            nj[k] = s_J[jj[k]];
#pragma unroll
            for (int w = 0; w < kMaskWords; ++w) nm[k][w] = s_anc[n][w] | s_anc[jj[k]][w];
          }
        }
      }
      __syncwarp();
#pragma unroll
      for (int k = 0; k < 3; ++k) {
        const int n = lane + 32 * k;
        if (n < N && jj[k] >= 0) {
          s_dep[n] = nd[k];
          s_J[n] = nj[k];
#pragma unroll
          for (int w = 0; w < kMaskWords; ++w) s_anc[n][w] = nm[k][w];
        }
      }
      __syncwarp();
    }
  }
  __syncthreads();   // barriers initialised, ctx known (unless pipelined)
  if (!p.pipelined) {
    C = s_C;
    derive();
  }
  // ---- Q: once the bf16 rows have landed, warps 1..15 convert them into
  // the fp16 swizzled tile in sQ; rows past the tile's are zero. No barrier
  // of its own: the staged rows (in sK) are read before the barrier that
  // precedes the first write into sK (the first chunk's K / V wait, or the
  // one before a chunk built otherwise), and sQ before the one before S.
  if (unit >= 0 && li >= 0) {
    if (!wait_bounded([&]() { return mbar_try_wait(bar_q, 0); }) && li == 0)
      report(p.status, DFV_DEV_TIMEOUT);
    const uint8_t* qs = smem + L::kQStage;
#pragma unroll 1
    for (int it = li; it < kRowsPerTile * (D / 8); it += kLoaders) {
      const int row = it / (D / 8), c = it % (D / 8);
      uint4 v = make_uint4(0u, 0u, 0u, 0u);
      if (row < rows_g)
        v = bf16x8_to_f16x8(*reinterpret_cast<const uint4*>(qs + static_cast<size_t>(row) * D * 2 + c * 16));
      *reinterpret_cast<uint4*>(sQ + tc::sw128_offset(row, c, kRowsPerTile)) = v;
    }
  }

  // ---- logits: CTAs without an attention unit scan their staged slices;
  // when nothing is staged, every CTA scans slices with plain loads
  auto accept_inputs = [&]() {
    if (lreg) scan_slices<LT>(p, lstage, ls0, lsn, bar_lg, &s_ok);
    if (!p.lbulk) plain_slices<LT>(p, blk, G);
    // ---- the walker keeps the tree's parents and tokens in smem
    if (blk == p.walker && tid < N) {
      s_wpar[tid] = p.parent[tid];
      s_wtok[tid] = p.tokens[tid];
    }
    // ---- pre-quantise tree rows: into the walker's own smem when it has no
    // attention unit and they fit, else into the workspace, spread over all
    // CTAs
    const int tot = N * p.hkv * 2 * NB;
    uint8_t* qdst = p.walker_local ? sK : p.qrows;
    const bool mine = p.walker_local ? blk == p.walker : true;
    if (mine) {
      const int nq = p.walker_local ? 1 : G;
      const int bq = p.walker_local ? 0 : blk;
      prequant_tree<D, FMT>(p, qdst, static_cast<int>(static_cast<long>(bq) * tot / nq),
                            static_cast<int>(static_cast<long>(bq + 1) * tot / nq));
    }
  };
  // pipelined: this reads only the step's own inputs and workspace, and runs
  // while the previous kernel finishes; ctx and the K / V copy come after it
  if (p.do_accept) accept_inputs();
  if (p.pipelined) {
    grid_dep_wait();
    if (tid == 0) {
      ctx_and_first_kv();
      if (p.do_accept && blk != p.walker && !late_signal) atomicAdd(p.bar + 2, 1u);
    }
    __syncthreads();
    C = s_C;
    derive();
  }

  if (late_signal) {
    __syncthreads();   // every thread's partials and tree rows written
    signal_done();
  }

  if (unit >= 0) {
    if (blk == 0 && tid < N && s_dep[tid] > p.max_depth) report(p.status, DFV_DEV_DEPTH);
    if (tid < kRowsPerTile) {
      const int rg = grp * kRowsPerTile + tid;
      if (rg < p.rows) {
        const int node = div_small(rg, p.group_m);
        s_row_node[tid] = node;
        s_row_lo[tid] = p.window > 0 ? C + s_dep[node] - p.window + 1 : 0;
      } else {
        s_row_node[tid] = -1;
        s_row_lo[tid] = 0x7fffffff;
      }
    }
    tc::fence_after_sync();

    const uint32_t tmem = *s_tmem;
    const uint32_t t_o = tmem + kChunk;           // O: columns [128, 128 + D)
    const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const int r = (warp & 3) * 32 + lane;   // this thread's row
    const int hc = warp >> 2;               // its quarter of the keys / of O's columns
    // A warp whose 32 rows all lie past the last row (a padded tile) skips
    // the second half of the softmax and the epilogue: its P rows are zero,
    // and its O rows reach no output.
    const bool live = grp * kRowsPerTile + (warp & 3) * 32 < p.rows;
    uint32_t ph_kv = 0, ph_s = 0, ph_pv = 0;
    int s_pend = 0, pv_pend = 0;   // thread 0: MMA batches issued, not yet waited for
    float m_run = -INFINITY, l_half = 0.f;
    bool o_valid = false, alive = true;
    const float sc = p.scale_log2;
    const int n_it = c1 - c0;
    bool last_seen = true;         // this thread saw the last chunk's P V done
    // Hand-off to warp 0 (named barrier 3): warp 0 waits until every thread
    // has arrived, the others arrive and go on. Two uses are always
    // separated by a full CTA barrier.
    auto to_warp0 = [&]() {
      if (warp == 0) named_sync(3, kStepThreads);
      else named_arrive(3, kStepThreads);
    };
    auto chunk_of = [&](int i) { return i < n_tree ? T - 1 : c0 + (i - n_tree); };
    // S of chunk i in TMEM columns [0, 128) or [384, 512) by parity (clear
    // of O); its P (fp16 pairs) overwrites the first 64 of them
    auto t_sbuf = [&](int i) { return tmem + ((i & 1) ? 384u : 0u); };

    // One operand of a committed chunk at key j0 (nk keys) into its swizzled
    // [keys][D] fp16 tile (kvi 0: K^ -> sK, 1: V^ -> sV).
    // binary16 rows: each thread copies 16-byte pieces straight into their
    // swizzled slots; rows past the chunk's keys are zero
    // (threads t0, t0 + 1, ... of nt take the pieces in turn)
    auto f16_copy = [&](int kvi, int j0, int nk, int t0, int nt) {
      constexpr int PR = D / 8;                           // pieces per row
      const uint8_t* b = (kvi ? p.v_cache : p.k_cache) + (static_cast<size_t>(h) * p.capacity + j0) * (D * 2);
      uint8_t* dst0 = kvi ? sV : sK;
#pragma unroll 1
      for (int it = t0; it < kChunk * PR; it += nt) {
        const int key = it / PR, c = it % PR;
        uint8_t* dst = dst0 + tc::sw128_offset(key, c, kChunk);
        if (key < nk) cp_async16(dst, b + key * (D * 2) + c * 16);
        else *reinterpret_cast<uint4*>(dst) = make_uint4(0u, 0u, 0u, 0u);
      }
      cp_async_wait_all();
    };
    // Q4_0 rows: a work item is a pair of blocks (36 bytes = 9 words, 64
    // elements = one swizzle block) of one key row. Within a warp, lanes
    // 8i..8i+7 take eight consecutive keys of the same pair: the 16-byte
    // stores of each 8-lane phase then fall on 8 distinct swizzled granules,
    // and the 9-word loads (word stride 9 * pairs-per-row between keys, 9
    // between pairs) fall on 32 distinct banks. `raw` is the rows' copy in
    // smem, or null to read them from the cache.
    // Item g (< HALF) of an operand; the thread of item g holds lane g % 32.
    constexpr int PPK = D / 64;                           // block pairs per key row
    constexpr int HALF = kChunk * PPK;                    // items per operand
    constexpr int kWorkers = kStepThreads - 32;           // warps 1.. (warp 0 issues the MMAs)
    static_assert(HALF <= 2 * kWorkers, "at most two dequant items per worker and operand");
    auto q4_pos = [&](int g, int& key, int& pp) {
      const int l = g & 31;
      key = (g >> 5) * (32 / PPK) + (l & 7) + 8 * (l / (8 * PPK));
      pp = (l >> 3) % PPK;
    };
    auto q4_load = [&](int g, int kvi, const uint8_t* raw, int j0, int nk, uint32_t* w) {
      int key, pp;
      q4_pos(g, key, pp);
      const bool on = g < HALF && key < nk;
      const uint8_t* base = raw != nullptr ? raw
          : (kvi ? p.v_cache : p.k_cache) + (static_cast<size_t>(h) * p.capacity + j0) * L::kRowB;
      const uint32_t* src = reinterpret_cast<const uint32_t*>(base + (on ? key * L::kRowB + pp * 36 : 0));
#pragma unroll
      for (int e = 0; e < 9; ++e) w[e] = on ? src[e] : 0u;
    };
    auto q4_store = [&](int g, int kvi, const uint32_t* w) {
      if (g < HALF) {
        int key, pp;
        q4_pos(g, key, pp);
        uint4 o4[8];
        q4_0_pair_chunks(w, o4);       // all-zero blocks dequantise to zeros
        uint8_t* dst = kvi ? sV : sK;
#pragma unroll
        for (int e = 0; e < 8; ++e)
          *reinterpret_cast<uint4*>(dst + tc::sw128_offset(key, pp * 8 + e, kChunk)) = o4[e];
      }
    };
    // the workers' K^ handed to warp 0: 0 when their wait for the raw rows
    // gave up
    __shared__ int s_wok;
    // S = Q K^T (M = 128 rows, N = 128 keys, K = D) into t_dst. The issue
    // loop is unrolled and each descriptor is the tile's first plus the
    // step's offset (16-byte units): a rolled loop that rebuilt them cost
    // the issuing thread about 40 % more time per MMA.
    auto issue_s = [&](uint32_t t_dst) {
      tc::fence_after_sync();
      constexpr uint32_t ida = tc::idesc_f16(kRowsPerTile, kChunk);
      const uint64_t qd = tc::smem_desc_sw128(smem_u32(sQ), 1024);
      const uint64_t kd = tc::smem_desc_sw128(smem_u32(sK), 1024);
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        const uint64_t off = static_cast<uint64_t>(((kk >> 2) * kRowsPerTile * 128 + (kk & 3) * 32) >> 4);
        tc::mma_f16(t_dst, qd + off, kd + off, ida, kk > 0 ? 1u : 0u);
      }
      tc::commit(bar_s);
      ++s_pend;
    };

    // ---- the first chunk: K^ and V^ together, then its S. Its raw rows
    // (Q4_0, bulk) were copied into sV at entry; the tree chunk is built
    // from the tree rows.
    if (n_it > 0) {
      const int cc = chunk_of(0);
      const bool committed = cc < n_cc;
      const int j0 = lo_min + cc * kChunk;
      const int nk = committed ? min(kChunk, C - j0) : 0;
      if (committed && !kQ4) {
        __syncthreads();   // the staged Q rows (in sK) are converted
        f16_copy(0, j0, nk, tid, kStepThreads);
        f16_copy(1, j0, nk, tid, kStepThreads);
      } else if (committed) {
        // every thread waits for the raw rows itself; the barrier after the
        // loads (raw rows consumed, staged Q rows converted) also makes the
        // outcome of the wait the same for all
        bool seen = true;
        if constexpr (L::kBulk) seen = mbar_wait_bounded(bar_kv, ph_kv);
        uint32_t wk[9], wv[9];
        q4_load(tid, 0, L::kBulk ? sV + L::kRawK : nullptr, j0, nk, wk);
        q4_load(tid, 1, L::kBulk ? sV + L::kRawV : nullptr, j0, nk, wv);
        alive = __syncthreads_and(seen) != 0;
        if (alive) {
          if constexpr (L::kBulk) {
            ph_kv ^= 1u;
            kv_pending = 0;
          }
          q4_store(tid, 0, wk);
          q4_store(tid, 1, wv);
        } else if (tid == 0) {
          report(p.status, DFV_DEV_TIMEOUT);
        }
      } else {
        __syncthreads();   // the staged Q rows (in sK) are converted
        // tree chunk: keys t = 0..N-1 from tree_k / tree_v (bf16 -> fp16);
        // the other key rows are zero. The first TP pieces of each loader
        // thread were loaded at entry.
        const int nt = nt_all;
        const int real = tree_real;
        if (kQ4 && p.tree_q) {
          // the tree rows as the commit stores them: each 32-value block is
          // quantised to Q4_0 (the commit's rule) and dequantised again
#pragma unroll 1
          for (int it = tid; it < 2 * nt * NB; it += kStepThreads) {
            const int ka = it / NB, b = it % NB;
            const int kvi = ka >= nt ? 1 : 0, key = ka - kvi * nt;
            const uint4* src = reinterpret_cast<const uint4*>(
                (kvi ? p.tree_v : p.tree_k) + (static_cast<size_t>(key) * p.hkv + h) * D + b * 32);
            float x[32];
#pragma unroll
            for (int u4 = 0; u4 < 4; ++u4) {
              const uint4 r4 = __ldg(src + u4);
              const __nv_bfloat162* hb = reinterpret_cast<const __nv_bfloat162*>(&r4);
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                const float2 f = __bfloat1622float2(hb[e]);
                x[u4 * 8 + 2 * e] = f.x;
                x[u4 * 8 + 2 * e + 1] = f.y;
              }
            }
            uint32_t code[4], dbits;
            q4_0_quantize_regs(x, code, dbits);
            uint4 o4[4];
            q4_0_block_chunks(code, dbits, o4);
#pragma unroll
            for (int e = 0; e < 4; ++e)
              *reinterpret_cast<uint4*>((kvi ? sV : sK) + tc::sw128_offset(key, b * 4 + e, kChunk)) = o4[e];
          }
        } else if (li >= 0) {
#pragma unroll
          for (int u = 0; u < TP; ++u) {
            const int it = li + u * kLoaders;
            if (it < real) {
              const int ka = it / (D / 8), c = it % (D / 8);
              const int kvi = ka >= nt ? 1 : 0, key = ka - kvi * nt;
              *reinterpret_cast<uint4*>((kvi ? sV : sK) + tc::sw128_offset(key, c, kChunk)) =
                  bf16x8_to_f16x8(tv[u]);
            }
          }
#pragma unroll 1
          for (int it = li + TP * kLoaders; it < real; it += kLoaders) {
            const int ka = it / (D / 8), c = it % (D / 8);
            const int kvi = ka >= nt ? 1 : 0, key = ka - kvi * nt;
            const uint4 v = __ldg(reinterpret_cast<const uint4*>(
                (kvi ? p.tree_v : p.tree_k) + (static_cast<size_t>(key) * p.hkv + h) * D + c * 8));
            *reinterpret_cast<uint4*>((kvi ? sV : sK) + tc::sw128_offset(key, c, kChunk)) =
                bf16x8_to_f16x8(v);
          }
        }
        const int zero = 2 * (kChunk - nt) * (D / 8);
#pragma unroll 1
        for (int it = tid; it < zero; it += kStepThreads) {
          const int ka = it / (D / 8), c = it % (D / 8);
          const int kvi = ka >= kChunk - nt ? 1 : 0, key = nt + ka - kvi * (kChunk - nt);
          *reinterpret_cast<uint4*>((kvi ? sV : sK) + tc::sw128_offset(key, c, kChunk)) =
              make_uint4(0, 0, 0, 0);
        }
      }
      fence_proxy_async_smem();
      to_warp0();   // K^ and V^ written: warp 0 issues S, the others go on to wait for it
      if (alive && tid == 0) issue_s(t_sbuf(0));
    }

    // ---- chunk i: its S is in flight. Softmax -> P (TMEM); P V(i) goes in
    // flight and, under it, K^ of chunk i + 1 is built and its S issued;
    // once P V(i) is done, V^ of chunk i + 1. The raw rows of chunk i + 1
    // are copied while chunk i's softmax runs.
#pragma unroll 1
    for (int i = 0; i < n_it && alive; ++i) {
      const int cc = chunk_of(i);
      const bool committed = cc < n_cc;
      const int j0 = lo_min + cc * kChunk;
      const int nk = committed ? min(kChunk, C - j0) : 0;
      const uint32_t t_sb = t_sbuf(i);
      // every thread waits for S itself; the row-max barrier below makes
      // the outcome the same for all
      const bool s_seen = mbar_wait_bounded(bar_s, ph_s);
      tc::fence_after_sync();
      // K^ is consumed: the next chunk's raw K / V go in flight (every chunk
      // after the first is committed)
      if constexpr (L::kBulk && kQ4) {
        if (tid == 0 && s_seen && i + 1 < n_it) issue_kv(chunk_of(i + 1), sK + L::kRawK2, smem + L::kRawV2);
      }

      // ---- masked softmax of the 128-row tile: four threads per row, 32
      // keys each, loaded from TMEM once
      {
        const int kb0 = hc * 32;
        float s[32];
        tc::ld32(t_sb + lane_base + kb0, s);
        const int node = s_row_node[r], lo = s_row_lo[r];
        float cm[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
        if (committed) {
          // visible keys of this row form the range [kmin, kmax)
          const int kmin = min(max(lo - j0, 0), kChunk) - kb0;
          const int kmax = (node >= 0 ? nk : 0) - kb0;
          if (kmin <= 0 && kmax >= 32) {
            // every key of this thread's slice is visible (no range test)
#pragma unroll
            for (int k = 0; k < 32; ++k) cm[k & 3] = fmaxf(cm[k & 3], s[k]);
          } else {
#pragma unroll
            for (int k = 0; k < 32; ++k) {
              const float x = (k >= kmin && k < kmax) ? s[k] : -INFINITY;
              s[k] = x;
              cm[k & 3] = fmaxf(cm[k & 3], x);
            }
          }
        } else {
          // tree keys t = 0..N-1 (N <= 65 < 128: one tree chunk); this
          // thread's keys are ancestor-mask word hc
          const uint32_t w = (node >= 0 && hc < kMaskWords) ? s_anc[node][hc] : 0u;
#pragma unroll
          for (int k = 0; k < 32; ++k) {
            const float x = ((w >> k) & 1u) ? s[k] : -INFINITY;
            s[k] = x;
            cm[k & 3] = fmaxf(cm[k & 3], x);
          }
        }
        s_pmax[hc][r] = fmaxf(fmaxf(cm[0], cm[1]), fmaxf(cm[2], cm[3]));
        if (!__syncthreads_and(s_seen)) {
          if (tid == 0) report(p.status, DFV_DEV_TIMEOUT);
          alive = false;
        } else {
          ph_s ^= 1u;
          s_pend = 0;
        }
        if (alive && live) {
          // the scale (> 0) is applied to the row max and inside the exp:
          // max(s) * sc is the max of the scaled scores
          const float cmax = fmaxf(fmaxf(s_pmax[0][r], s_pmax[1][r]), fmaxf(s_pmax[2][r], s_pmax[3][r])) * sc;
          float alpha = 1.f;
          bool rescale = false;
          if (m_run == -INFINITY) {
            m_run = cmax;                       // O and l are still zero
          } else if (cmax > m_run + kRescaleLog2) {
            alpha = tc::ex2(m_run - cmax);
            rescale = true;
            m_run = cmax;
          }
          const float sub = m_run == -INFINITY ? 0.f : m_run;
          // P of this thread's 32 keys as 16 fp16 pairs over its S columns
          // (every S load of the tile precedes the barrier above)
          float rs4[4] = {0.f, 0.f, 0.f, 0.f};
          uint32_t pw[16];
#pragma unroll
          for (int k2 = 0; k2 < 16; ++k2) {
            const float p0 = tc::ex2(fmaf(s[2 * k2], sc, -sub));
            const float p1 = tc::ex2(fmaf(s[2 * k2 + 1], sc, -sub));
            rs4[k2 & 3] += p0 + p1;
            pw[k2] = pack_half2(p0, p1);
          }
          tc::st16(t_sb + lane_base + hc * 16, pw);
          l_half = l_half * alpha + ((rs4[0] + rs4[1]) + (rs4[2] + rs4[3]));
          if (o_valid && __any_sync(0xffffffffu, rescale)) {
            // this warp's quarter of the row's O columns
#pragma unroll 1
            for (int b = 0; b < D / 32; ++b) {
              const uint32_t col = static_cast<uint32_t>(hc * (D / 4) + b * 8);
              float ov[8];
              tc::ld8(t_o + lane_base + col, ov);
#pragma unroll
              for (int e = 0; e < 8; ++e) ov[e] *= alpha;
              tc::st8(t_o + lane_base + col, ov);
            }
          }
        } else if (alive) {
          // rows past the last: zero P (their O rows reach no output)
          uint32_t pw[16];
#pragma unroll
          for (int k2 = 0; k2 < 16; ++k2) pw[k2] = 0u;
          tc::st16(t_sb + lane_base + hc * 16, pw);
        }
      }
      if (!alive) break;   // S timed out (the same for every thread)
      tc::fence_before_sync();
      to_warp0();   // P written: warp 0 issues P V, the others go on

      // ---- O += P V (M = 128 rows, N = D, K = 128 keys; P from TMEM, V
      // MN-major)
      if (tid == 0) {
        tc::fence_after_sync();
        constexpr uint32_t ida = tc::idesc_f16(kRowsPerTile, D, true);
        const uint64_t vd = tc::smem_desc_sw128_mn(smem_u32(sV), kChunk * 128, 1024);
#pragma unroll
        for (int kk = 0; kk < kChunk / 16; ++kk)
          tc::mma_f16_ts(t_o, t_sb + static_cast<uint32_t>(kk * 8),
                         vd + static_cast<uint64_t>((kk * 16 * 128) >> 4), ida,
                         (o_valid || kk > 0) ? 1u : 0u);
        tc::commit(bar_mma);
        ++pv_pend;
      }
      if (i + 1 < n_it) {
        // The next chunk, by the workers (warps 1..) while warp 0 issues:
        // K^ under P V(i) (P is in TMEM, sK is free), handed to warp 0 for
        // its S; V^ once P V(i) has read sV. Warp 0's MMA issue may block
        // while the tensor pipe is busy; the workers do not wait for it.
        const int cn = chunk_of(i + 1);
        const int jn = lo_min + cn * kChunk;
        const int nn = min(kChunk, C - jn);
        if (tid == 32) s_wok = 1;   // (the F16 and unstaged paths have no copy to wait on)
        bool ok = true;             // a worker: every wait of this chunk ended in time
        if (warp == 0) {
          __syncwarp();
          named_sync(2, kStepThreads);              // K^ written (or a wait gave up)
          if (tid == 0 && s_wok) issue_s(t_sbuf(i + 1));
          __syncwarp();
        } else {
          // every worker waits on the copy and on P V itself; the barriers
          // that follow carry the outcome to all
          const int wi = tid - 32;
          if constexpr (!kQ4) {
            f16_copy(0, jn, nn, wi, kWorkers);
          } else {
            bool seen = true;
            if constexpr (L::kBulk) seen = mbar_wait_bounded(bar_kv, ph_kv);
            uint32_t wk[9], wk2[9];
            q4_load(wi, 0, L::kBulk ? sK + L::kRawK2 : nullptr, jn, nn, wk);
            q4_load(wi + kWorkers, 0, L::kBulk ? sK + L::kRawK2 : nullptr, jn, nn, wk2);
            if constexpr (L::kBulk) {
              ok = named_sync_and(1, kWorkers, seen);   // raw K (in sK) consumed
              if (!ok && tid == 32) report(p.status, DFV_DEV_TIMEOUT);
            }
            if (tid == 32) s_wok = ok ? 1 : 0;
            if (ok) {
              q4_store(wi, 0, wk);
              q4_store(wi + kWorkers, 0, wk2);
            }
          }
          fence_proxy_async_smem();
          named_arrive(2, kStepThreads);
          if (ok) {
            ok = mbar_wait_bounded(bar_mma, ph_pv);
            if (!ok) report(p.status, DFV_DEV_TIMEOUT);
          }
          if (ok) {
            if constexpr (!kQ4) {
              f16_copy(1, jn, nn, wi, kWorkers);
            } else {
              uint32_t wv[9], wv2[9];
              q4_load(wi, 1, L::kBulk ? smem + L::kRawV2 : nullptr, jn, nn, wv);
              q4_load(wi + kWorkers, 1, L::kBulk ? smem + L::kRawV2 : nullptr, jn, nn, wv2);
              q4_store(wi, 1, wv);
              q4_store(wi + kWorkers, 1, wv2);
            }
            fence_proxy_async_smem();
          }
        }
        // V^ written, S issued; false if any wait gave up
        if (!__syncthreads_and(warp == 0 || ok)) { alive = false; break; }
        if constexpr (kQ4 && L::kBulk) {
          ph_kv ^= 1u;
          kv_pending = 0;
        }
        ph_pv ^= 1u;                                // P V(i) is done
        pv_pend = 0;
        o_valid = true;
        tc::fence_after_sync();
      } else {
        // the last chunk: every thread waits for P V itself; the
        // epilogue's first barrier makes the outcome the same for all
        last_seen = mbar_wait_bounded(bar_mma, ph_pv);
        tc::fence_after_sync();
      }
    }
    // a unit that gave up waits (bounded) for its copies and MMAs still in
    // flight before its smem and TMEM are reused or released
    if (!alive && tid == 0) {
      if (kv_pending > 0) mbar_wait_bounded(bar_kv, ph_kv);
      if (pv_pend > 0) mbar_wait_bounded(bar_mma, ph_pv);
      if (s_pend > 0) mbar_wait_bounded(bar_s, ph_s);
    }

    // ---- epilogue: normalised O rows from TMEM (each thread's columns in
    // one batch of loads) -> the unit's partial rows staged in smem (D fp16
    // values, then the row's (max, sum), 16 bytes more per row) -> one bulk
    // copy to the workspace; or straight to the output (fp32) when there is
    // one split
    s_l[hc][r] = l_half;
    const bool pv_all = __syncthreads_and(last_seen) != 0;
    if (n_it > 0 && alive) {
      if (pv_all) {
        ph_pv ^= 1u;
        pv_pend = 0;
        o_valid = true;
      } else {
        alive = false;
        if (tid == 0) {
          report(p.status, DFV_DEV_TIMEOUT);
          mbar_wait_bounded(bar_mma, ph_pv);   // the MMAs still in flight (bounded)
        }
      }
    }
    const bool ok_all = o_valid && alive;
    constexpr int RB = kPartRowBytes<D>;   // bytes of one partial row
    uint8_t* stage = smem;                 // [rows_g][RB], over sQ and sK (free after the last MMA)
    if (ok_all && live) {
      // the TMEM loads are warp-wide (.sync.aligned): every lane loads, the
      // lanes of real rows store
      const bool mine = r < rows_g;
      const float l = (s_l[0][r] + s_l[1][r]) + (s_l[2][r] + s_l[3][r]);
      const float inv = l > 0.f ? __fdividef(1.f, l) : 0.f;
      constexpr int CT = D / 4;            // columns of this thread
      float ov[CT];
      const uint32_t col0 = t_o + lane_base + hc * CT;
      if constexpr (CT == 64) tc::ld32x2(col0, col0 + 32, ov);
      else if constexpr (CT == 32) tc::ld32(col0, ov);
      else tc::ld16(col0, ov);
      if (mine) {
        const int rg = grp * kRowsPerTile + r;
        const int node = div_small(rg, p.group_m), qh = h * p.group + rg - node * p.group;
        if (p.splits == 1) {
          float4* dst = reinterpret_cast<float4*>(p.out + (static_cast<size_t>(node) * p.hq + qh) * D + hc * CT);
#pragma unroll
          for (int e = 0; e < CT / 4; ++e)
            dst[e] = make_float4(ov[4 * e] * inv, ov[4 * e + 1] * inv, ov[4 * e + 2] * inv, ov[4 * e + 3] * inv);
          if (hc == 0 && p.lse != nullptr) p.lse[node * p.hq + qh] = (m_run + log2f(l)) * 0.69314718055994531f;
        } else {
          uint4* dst = reinterpret_cast<uint4*>(stage + r * RB + hc * CT * 2);
#pragma unroll
          for (int e = 0; e < CT / 8; ++e)
            dst[e] = make_uint4(pack_half2(ov[8 * e] * inv, ov[8 * e + 1] * inv),
                                pack_half2(ov[8 * e + 2] * inv, ov[8 * e + 3] * inv),
                                pack_half2(ov[8 * e + 4] * inv, ov[8 * e + 5] * inv),
                                pack_half2(ov[8 * e + 6] * inv, ov[8 * e + 7] * inv));
          if (hc == 0)
            *reinterpret_cast<float2*>(stage + r * RB + D * 2) = make_float2(l > 0.f ? m_run : -INFINITY, l);
        }
      }
    }
    tc::fence_before_sync();
    fence_proxy_async_smem();   // the staged rows, before the bulk copy reads them
    to_warp0();   // warp 0 copies the partials out and frees TMEM; the others go on
    if (p.splits > 1) {
      uint8_t* part = p.part + static_cast<size_t>(unit) * kRowsPerTile * RB;
      if (!ok_all) {
        // a timed-out unit publishes empty rows (max -inf, sum 0): the merge
        // leaves it out (the status reports the timeout)
        if (tid < rows_g)
          *reinterpret_cast<float2*>(part + tid * RB + D * 2) = make_float2(-INFINITY, 0.f);
        __syncthreads();
      }
      if (tid == 0) {
        if (ok_all) {
          bulk_s2g(part, stage, static_cast<uint32_t>(rows_g * RB));
          bulk_commit_wait();
        }
        // The split group's word: each CTA adds 1 (low 16 bits: arrivals;
        // high 16 bits: a generation); the last to arrive adds 2^16 - n,
        // which clears the count and advances the generation for the next
        // launch. Every CTA of the group reads the same generation g from its
        // own add and marks its partial written with (g + 1) mod 2^16.
        const unsigned int n = static_cast<unsigned int>(p.splits);
        if ((arrive_old & 0xFFFFu) == n - 1) atomicAdd(p.bar + 4 + 2 * (unit / p.splits), 0x10000u - n);
        s_tag = ((arrive_old >> 16) + 1u) & 0xFFFFu;
        fence_proxy_async_global();   // the bulk writes, before the generic release below
        __threadfence();              // the CTA's partial rows before its ready word
        asm volatile("st.relaxed.gpu.global.u32 [%0], %1;" ::"l"(p.ready + unit), "r"(s_tag) : "memory");
      }
    }
    if (warp == 0) tc::tmem_dealloc(tmem, kTmemCols);
  }
  // ---- the walker: once every other CTA has read ctx and written its
  // argmax partial, merge the partials, walk and commit -- all before the
  // group barriers, under the attention of the other CTAs
  if (p.do_accept && blk == p.walker) walker_tail<D, FMT>(p, G, C, s_ctx_ok != 0, sQ, sK, s_wpar, s_wtok);

  // ================================================================ merge
  // Each of the `splits` CTAs of a (KV head, tile group) group waits for the
  // group's partials to be marked ready, then merges its share of the
  // group's rows over the splits by log-sum-exp: the rows (values, max and
  // sum) of every split's partial arrive by one bulk copy per split into
  // smem, where each thread merges four columns of one row.
  if (unit >= 0 && p.splits > 1) {
    constexpr int RB = kPartRowBytes<D>;
    const int gi = unit / p.splits, split_ = unit % p.splits;
    const int h_ = gi / p.n_grp, g_ = gi % p.n_grp;
    const int rows_t = min(kRowsPerTile, p.rows - g_ * kRowsPerTile);
    const int r0 = split_ * rows_t / p.splits, r1 = (split_ + 1) * rows_t / p.splits;
    const int nr = r1 - r0, S = p.splits;
    if (nr <= 0) return;
    const size_t ubase = static_cast<size_t>(gi) * S;
    uint8_t* mst = sK;   // [S][nr][RB]
    if (blk == p.walker) __syncthreads();   // (a walker with a unit: its copies out of sK are done)
    // Warp 0 waits for the group's ready words and lane 0 then starts the
    // copies; the other threads only wait for the copies to land (no CTA
    // barrier between). If the ready wait gives up, no copy starts and
    // every thread's own wait runs out and returns.
    if (warp == 0) {
      __syncwarp();   // s_tag was written by lane 0
      const bool ok = wait_ready(p.ready + static_cast<size_t>(gi) * p.splits, p.splits, s_tag);
      if (lane == 0) {
        if (ok) {
          fence_proxy_async_global();   // the acquired partials, before the async-proxy reads
          mbar_arrive_expect_tx(bar_q, static_cast<uint32_t>(S * nr * RB));
          for (int s = 0; s < S; ++s)
            bulk_g2s(mst + static_cast<size_t>(s) * nr * RB, p.part + ((ubase + s) * kRowsPerTile + r0) * RB,
                     static_cast<uint32_t>(nr * RB), bar_q);
        } else {
          report(p.status, DFV_DEV_TIMEOUT);
        }
      }
      if (!ok) return;
    }
    if (!wait_bounded([&]() { return mbar_try_wait(bar_q, 1); })) {
      if (tid == 32) report(p.status, DFV_DEV_TIMEOUT);
      return;
    }
    // Each thread merges four columns of one row over the splits; every
    // thread of a row derives the row's weights from the staged (max, sum)
    // tails itself, so no phase or barrier separates weights and sums.
    constexpr int PR = D / 4;                       // four-column pieces per row
#pragma unroll 1
    for (int it = tid; it < nr * PR; it += kStepThreads) {
      const int rr = it / PR, c = it % PR;
      const uint8_t* row0 = mst + static_cast<size_t>(rr) * RB;
      const size_t sstride = static_cast<size_t>(nr) * RB;   // bytes between splits' rows
      float M = -INFINITY;
#pragma unroll 4
      for (int sp = 0; sp < S; ++sp) M = fmaxf(M, reinterpret_cast<const float2*>(row0 + sp * sstride + D * 2)->x);
      float lsum = 0.f, acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 2
      for (int sp = 0; sp < S; ++sp) {
        const float2 t = *reinterpret_cast<const float2*>(row0 + sp * sstride + D * 2);
        const float w = t.x == -INFINITY ? 0.f : tc::ex2(t.x - M) * t.y;
        lsum += w;
        const uint2 v = *reinterpret_cast<const uint2*>(row0 + sp * sstride + c * 8);
        const float2 f0 = __half22float2(*reinterpret_cast<const __half2*>(&v.x));
        const float2 f1 = __half22float2(*reinterpret_cast<const __half2*>(&v.y));
        acc[0] += w * f0.x;
        acc[1] += w * f0.y;
        acc[2] += w * f1.x;
        acc[3] += w * f1.y;
      }
      const float inv = lsum > 0.f ? 1.f / lsum : 0.f;
      const int rg = g_ * kRowsPerTile + r0 + rr;
      const int node = div_small(rg, p.group_m), qh = h_ * p.group + rg - node * p.group;
      *reinterpret_cast<float4*>(p.out + (static_cast<size_t>(node) * p.hq + qh) * D + c * 4) =
          make_float4(acc[0] * inv, acc[1] * inv, acc[2] * inv, acc[3] * inv);
      if (c == 0 && p.lse != nullptr) p.lse[node * p.hq + qh] = (M + log2f(lsum)) * 0.69314718055994531f;
    }
  }
}

// ---------------------------------------------------------------- host side

static size_t a256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

static bool step_plan(int n_nodes, int hq, int hkv, int head_dim, int window, int cap, int vocab,
                      int logits_dtype, bool with_accept, int kv_fmt, StepPlan* pl) {
  if (n_nodes < 1 || n_nodes > kMaxNodes || hkv < 1 || hq < hkv || hq % hkv || hq > 256 ||
      window < 0 || cap < 0)
    return false;
  if (head_dim != 64 && head_dim != 128 && head_dim != 256) return false;
  if (with_accept && vocab < 1) return false;
  const int sms = sm_count();
  pl->grid = sms < kMaxStepGrid ? sms : kMaxStepGrid;
  pl->rows = n_nodes * (hq / hkv);
  pl->n_grp = (pl->rows + kRowsPerTile - 1) / kRowsPerTile;   // 128-row tiles per KV head
  const long groups = static_cast<long>(hkv) * pl->n_grp;
  if (groups > pl->grid) return false;                  // more (head, group) pairs than SMs
  const long kbound = window > 0 ? (window - 1 < cap ? window - 1 : cap) : cap;
  const long tb = (kbound + kChunk - 1) / kChunk + (n_nodes + kChunk - 1) / kChunk;
  // one chunk per split when that leaves a CTA for the walker; otherwise (long
  // contexts) every split takes several chunks and a few CTAs stay for the
  // logits
  long s;
  if (groups * tb <= pl->grid - (with_accept ? 1 : 0)) {
    s = tb;
  } else if (!with_accept) {
    s = pl->grid / groups;
  } else {
    // Keep `keep` CTAs out of the attention (the walker and keep - 1 that
    // scan the logits): the count that minimises the longer of the two
    // estimated paths, a unit's chunks at kChunkCostNs each and a spare's
    // share of the logits at kSpareBytesPerUs (both measured on a GB300
    // over budgets 22 to 64); ties go to the fewer spares.
    const long lbytes = static_cast<long>(n_nodes) * vocab * (logits_dtype == DFV_DTYPE_BF16 ? 2 : 4);
    long best = -1, best_cost = 0;
    for (long keep = 2; keep <= pl->grid - groups; ++keep) {
      const long sk = (pl->grid - keep) / groups;
      const long attn = (tb + sk - 1) / sk * kChunkCostNs;
      const long lg = lbytes * 1000 / ((keep - 1) * kSpareBytesPerUs);
      const long cost = attn > lg ? attn : lg;
      if (best < 0 || cost < best_cost) {
        best = keep;
        best_cost = cost;
      }
    }
    s = (pl->grid - best) / groups;
  }
  if (s > kMaxStepSplits) s = kMaxStepSplits;
  {
    // the merge stages every split's share of a group's rows in sK + sV:
    // at most (rows + splits) rows of D fp16
    long merge_b;
    switch (head_dim) {
      case 64: merge_b = StepSmem<64>::kKBytes + kChunk * 64 * 2; break;
      case 128: merge_b = StepSmem<128>::kKBytes + kChunk * 128 * 2; break;
      default: merge_b = StepSmem<256>::kKBytes + kChunk * 256 * 2; break;
    }
    while (s > 1 && (kRowsPerTile + s) * (head_dim * 2 + 16) > merge_b) --s;
  }
  if (s < 1) return false;
  pl->splits = static_cast<int>(s);
  pl->units = static_cast<int>(groups) * pl->splits;
  const int tile_b = kRowsPerTile * head_dim * 2;
  // the walker stages every argmax partial in its Q tile
  const int max_parts = tile_b / static_cast<int>(sizeof(ArgPartial));
  const int esz = logits_dtype == DFV_DTYPE_BF16 ? 2 : 4;
  // the walker: a CTA without an attention unit when there is one
  pl->walker = with_accept ? (pl->grid > pl->units ? pl->grid - 1 : 0) : -1;
  for (int i = 0; i < kMaxStepGrid; ++i) pl->lslot[i] = 0u;
  pl->lchunks = pl->lunits = pl->lchunk_len = pl->lbulk = pl->lstride = pl->lper = 0;
  if (with_accept) {
    // Logits slices are staged (bulk copies into smem) on the CTAs without an
    // attention unit, the walker aside, in rounds through the two halves of
    // their staging area (a round: the slices one half holds). The slice
    // count per node is the one whose even share puts the least work
    // (bytes plus a fixed cost per slice) on each of those CTAs. Otherwise
    // every CTA scans slices with plain loads.
    const int cap_c = (vocab + 255) / 256;
    int spare_b;
    switch (head_dim) {
      case 64: spare_b = StepSmem<64>::kSpareStageBytes; break;
      case 128: spare_b = StepSmem<128>::kSpareStageBytes; break;
      default: spare_b = StepSmem<256>::kSpareStageBytes; break;
    }
    int unit_b;
    switch (head_dim) {
      case 64: unit_b = StepSmem<64>::kUnitStageBytes; break;
      case 128: unit_b = StepSmem<128>::kUnitStageBytes; break;
      default: unit_b = StepSmem<256>::kUnitStageBytes; break;
    }
    // light units: the splits of a last tile of at most kLightRows real
    // rows (no remainder folded in); they stage one round at entry and scan
    // it while their K / V chunk is still in flight
    int spare[kMaxStepGrid], nsp = 0, light[kMaxStepGrid], nlu = 0;
    const int last_rows = pl->rows - (pl->n_grp - 1) * kRowsPerTile;
    if (pl->n_grp > 1 && last_rows <= kLightRows)
      for (int u = 0; u < pl->units; ++u)
        if ((u / pl->splits) % pl->n_grp == pl->n_grp - 1 && u != pl->walker) light[nlu++] = u;
    for (int b = pl->units; b < pl->grid; ++b)
      if (b != pl->walker) spare[nsp++] = b;
    const int align_el = 16 / esz;
    int best_lc = -1, best_len = 0, best_per = 0, best_lu = 0;
    long best_load = 0;
    if (nsp + nlu > 0 && static_cast<long>(vocab) * esz % 16 == 0) {
      const int max_lc = cap_c < max_parts / n_nodes ? cap_c : max_parts / n_nodes;
      for (int lc = 1; lc <= max_lc; ++lc) {
        const int len = (((vocab + lc - 1) / lc) + align_el - 1) / align_el * align_el;
        const long sb = static_cast<long>(len) * esz;
        long per = (spare_b / 2) / sb;
        if (per > kMaxStagedSlices / 2) per = kMaxStagedSlices / 2;
        const long per_u = nlu > 0 ? (unit_b / sb < per ? unit_b / sb : per) : 0;
        const long need = static_cast<long>(n_nodes) * lc;
        const long lu = need < nlu * per_u ? need : nlu * per_u;   // slices on light units
        const long rest = need - lu;
        if (rest > 0 && (nsp == 0 || per < 1)) continue;
        if (lu == 0 && per < 1) continue;
        const long spare_load = nsp > 0 ? (rest + nsp - 1) / nsp * (sb + kSliceCostBytes) : 0;
        const long lu_load = nlu > 0 ? (lu + nlu - 1) / nlu * (sb + kSliceCostBytes) : 0;
        const long load = spare_load > lu_load ? spare_load : lu_load;
        if (best_lc < 0 || load < best_load) {
          best_lc = lc;
          best_len = len;
          best_per = static_cast<int>(per < 1 ? 1 : per);
          best_lu = static_cast<int>(lu);
          best_load = load;
        }
      }
    }
    if (best_lc > 0) {
      pl->lchunks = best_lc;
      pl->lunits = n_nodes * best_lc;
      pl->lchunk_len = best_len;
      pl->lstride = best_len * esz;
      pl->lper = best_per;
      pl->lbulk = 1;
      int sl = 0;
      for (int i = 0; i < nlu && sl < best_lu; ++i) {
        const int c = best_lu / nlu + (i < best_lu % nlu ? 1 : 0);
        if (c > 0) {
          pl->lslot[light[i]] = static_cast<uint32_t>(sl) | (static_cast<uint32_t>(c) << 16);
          sl += c;
        }
      }
      const int rest = pl->lunits - sl;
      for (int i = 0; i < nsp && sl < pl->lunits; ++i) {
        const int c = rest / nsp + (i < rest % nsp ? 1 : 0);
        if (c > 0) {
          pl->lslot[spare[i]] = static_cast<uint32_t>(sl) | (static_cast<uint32_t>(c) << 16);
          sl += c;
        }
      }
    } else {
      // plain loads: CTA b takes slices b, b + grid, ...
      const int lim = kLogitVecs * kStepThreads * 16 < tile_b ? kLogitVecs * kStepThreads * 16 : tile_b;
      const int per_l = lim / esz;
      const int need_l = (vocab + per_l - 1) / per_l;
      int lc = pl->grid / n_nodes;
      if (lc < need_l) lc = need_l;
      if (lc > cap_c) lc = cap_c < need_l ? need_l : cap_c;
      if (lc > max_parts / n_nodes) lc = max_parts / n_nodes;   // longer slices instead
      pl->lchunks = lc;
      pl->lunits = n_nodes * lc;
      pl->lchunk_len = (((vocab + lc - 1) / lc) + align_el - 1) / align_el * align_el;
    }
  }
  int kbytes;
  switch (head_dim) {
    case 64: pl->smem = StepSmem<64>::kBytes; kbytes = StepSmem<64>::kKBytes; break;
    case 128: pl->smem = StepSmem<128>::kBytes; kbytes = StepSmem<128>::kKBytes; break;
    default: pl->smem = StepSmem<256>::kBytes; kbytes = StepSmem<256>::kKBytes; break;
  }
  {
    const long qbytes = static_cast<long>(n_nodes) * hkv * 2 * kv_row_bytes(kv_fmt, head_dim);
    pl->walker_local = with_accept && pl->grid > pl->units && qbytes <= kbytes ? 1 : 0;
  }
  // staged tree rows: sized for the larger (binary16) row, so one workspace
  // serves either cache format
  const int rowb = kv_row_bytes(DFV_KV_F16, head_dim);
  pl->ws_bar = 0;
  pl->ws_arg = a256(static_cast<size_t>(4 + 2 * groups + pl->units) * sizeof(unsigned int));
  pl->ws_qrows = pl->ws_arg + a256(static_cast<size_t>(pl->lunits) * sizeof(ArgPartial));
  pl->ws_ml = pl->ws_qrows + a256(with_accept ? static_cast<size_t>(n_nodes) * hkv * 2 * rowb : 0);
  const size_t nrow = pl->splits > 1 ? static_cast<size_t>(pl->units) * kRowsPerTile : 0;
  pl->ws_o = pl->ws_ml;
  pl->ws_total = pl->ws_o + a256(nrow * static_cast<size_t>(head_dim * 2 + 16));
  return true;
}

// A plain step is a cooperative launch (all CTAs resident at once). A
// pipelined one is launched with programmatic stream serialisation instead:
// its CTAs start on the SMs the previous kernel frees and wait in the kernel
// (griddepcontrol.wait) before touching ctx, the cache or the outputs. Its
// CTAs still all become resident, as the previous kernel never waits on
// them; and as each CTA takes a whole SM (one per SM: the register file),
// the step after it can only start once the one before it has completed,
// which is why two workspaces, used in turn, suffice.
template <int D, typename LT, int FMT>
static dfv_status step_launch_dt(StepParams& p, const StepPlan& pl, cudaStream_t stream) {
  static int configured[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return DFV_ERR_CUDA;
  if (!configured[dev]) {
    if (cudaFuncSetAttribute(step_kernel<D, LT, FMT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             StepSmem<D>::kBytes) != cudaSuccess)
      return DFV_ERR_CUDA;
    // exactly one CTA per SM: each holds all of the SM's TMEM columns
    int nb = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&nb, step_kernel<D, LT, FMT>, kStepThreads,
                                                      StepSmem<D>::kBytes) != cudaSuccess ||
        nb != 1)
      return DFV_ERR_CUDA;
    configured[dev] = 1;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(pl.grid);
  cfg.blockDim = dim3(kStepThreads);
  cfg.dynamicSmemBytes = StepSmem<D>::kBytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  if (p.pipelined) {
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
  } else {
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
  }
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, step_kernel<D, LT, FMT>, p) == cudaSuccess ? DFV_OK : DFV_ERR_CUDA;
}

// One instantiation per logits element type (the attention-only launch has
// no logits and takes the bf16 one).
template <int D, int FMT>
static dfv_status step_launch_f(StepParams& p, const StepPlan& pl, cudaStream_t stream) {
  if (p.do_accept && p.logits_dtype == DFV_DTYPE_F32) return step_launch_dt<D, float, FMT>(p, pl, stream);
  return step_launch_dt<D, __nv_bfloat16, FMT>(p, pl, stream);
}

template <int D>
static dfv_status step_launch_d(StepParams& p, const StepPlan& pl, int fmt, cudaStream_t stream) {
  if (fmt == DFV_KV_F16) return step_launch_f<D, DFV_KV_F16>(p, pl, stream);
  return step_launch_f<D, DFV_KV_Q4_0>(p, pl, stream);
}

// Workspace of either logits element size (the slicing differs slightly).
size_t step_workspace_bytes(int n_nodes, int hq, int hkv, int head_dim, int window, int cap,
                            int vocab, bool with_accept) {
  StepPlan a, b;
  if (!step_plan(n_nodes, hq, hkv, head_dim, window, cap, vocab, DFV_DTYPE_F32, with_accept,
                 DFV_KV_Q4_0, &a))
    return 0;
  step_plan(n_nodes, hq, hkv, head_dim, window, cap, vocab, DFV_DTYPE_BF16, with_accept, DFV_KV_Q4_0,
            &b);
  return a.ws_total > b.ws_total ? a.ws_total : b.ws_total;
}

// Attention only (with_accept = false) or the whole step.
dfv_status step_launch(bool with_accept, int n_nodes, int max_depth, int hq, int hkv,
                       int head_dim, int window, int kv_format, int cap, int vocab,
                       int logits_dtype, int32_t* ctx_len, void* k_cache, void* v_cache,
                       const void* q, const void* tree_k, const void* tree_v,
                       const int32_t* parent, const int32_t* tokens, const void* logits,
                       float scale, float* out, float* lse, int32_t* argmax, int32_t* accept_len,
                       int32_t* path, int32_t* out_tokens, void* workspace, size_t ws_bytes,
                       uint32_t* status, cudaStream_t stream) {
  const int fmt = kv_format & 0xFF, flags = kv_format & ~0xFF;
  if ((fmt != DFV_KV_Q4_0 && fmt != DFV_KV_F16) ||
      (flags & ~(DFV_KV_TREE_AS_CACHE | DFV_STEP_PIPELINED)) != 0)
    return DFV_ERR_UNSUPPORTED;
  if (head_dim != 64 && head_dim != 128 && head_dim != 256) return DFV_ERR_UNSUPPORTED;
  if (with_accept && logits_dtype != DFV_DTYPE_F32 && logits_dtype != DFV_DTYPE_BF16)
    return DFV_ERR_UNSUPPORTED;
  StepPlan pl;
  if (!step_plan(n_nodes, hq, hkv, head_dim, window, cap, vocab,
                 with_accept ? logits_dtype : DFV_DTYPE_F32, with_accept, fmt, &pl))
    return DFV_ERR_INVALID;
  if (!ctx_len || !k_cache || !v_cache || !q || !tree_k || !tree_v || !parent || !out || !workspace)
    return DFV_ERR_INVALID;
  if (with_accept && (!tokens || !logits || !argmax || !accept_len || !path || !out_tokens))
    return DFV_ERR_INVALID;
  if (!aligned(k_cache, 16) || !aligned(v_cache, 16) || !aligned(q, 16) || !aligned(tree_k, 16) ||
      !aligned(tree_v, 16) || !aligned(out, 16) || !aligned(workspace, 256) ||
      (with_accept && !aligned(logits, 16)))
    return DFV_ERR_INVALID;
  if (ws_bytes < pl.ws_total) return DFV_ERR_WORKSPACE;
  // pipelined: one CTA on every SM (see step_launch_dt)
  if ((flags & DFV_STEP_PIPELINED) && pl.grid != sm_count()) return DFV_ERR_UNSUPPORTED;
  StepParams p;
  p.n_nodes = n_nodes;
  p.max_depth = max_depth;
  p.hq = hq;
  p.hkv = hkv;
  p.group = hq / hkv;
  p.group_m = p.group == 1 ? 0u : static_cast<uint32_t>(((1ull << 32) + p.group - 1) / p.group);
  p.window = window;
  p.capacity = cap;
  p.vocab = vocab;
  p.logits_dtype = logits_dtype;
  p.rows = pl.rows;
  p.n_grp = pl.n_grp;
  p.splits = pl.splits;
  p.units = pl.units;
  p.lunits = pl.lunits;
  p.lchunks = pl.lchunks;
  p.lchunk_len = pl.lchunk_len;
  p.lbulk = pl.lbulk;
  p.lstride = pl.lstride;
  p.lper = pl.lper;
  p.do_accept = with_accept ? 1 : 0;
  // binary16 tree rows are exact in the cache format, so the flag only
  // changes anything for Q4_0
  p.tree_q = (flags & DFV_KV_TREE_AS_CACHE) && fmt == DFV_KV_Q4_0 ? 1 : 0;
  p.pipelined = (flags & DFV_STEP_PIPELINED) ? 1 : 0;
  p.walker = pl.walker;
  p.walker_local = pl.walker_local;
  for (int i = 0; i < kMaxStepGrid; ++i) p.lslot[i] = pl.lslot[i];
  const float sc = scale > 0.f ? scale : 1.0f / sqrtf(static_cast<float>(head_dim));
  p.scale_log2 = sc * 1.4426950408889634f;
  p.ctx_len = ctx_len;
  p.k_cache = static_cast<uint8_t*>(k_cache);
  p.v_cache = static_cast<uint8_t*>(v_cache);
  p.q = static_cast<const __nv_bfloat16*>(q);
  p.tree_k = static_cast<const __nv_bfloat16*>(tree_k);
  p.tree_v = static_cast<const __nv_bfloat16*>(tree_v);
  p.parent = parent;
  p.tokens = tokens;
  p.logits = logits;
  p.out = out;
  p.lse = lse;
  p.argmax = argmax;
  p.accept_len = accept_len;
  p.path = path;
  p.out_tokens = out_tokens;
  char* ws = static_cast<char*>(workspace);
  p.bar = reinterpret_cast<unsigned int*>(ws + pl.ws_bar);
  p.ready = p.bar + 4 + 2 * hkv * pl.n_grp;
  p.arg_part = reinterpret_cast<ArgPartial*>(ws + pl.ws_arg);
  p.qrows = reinterpret_cast<uint8_t*>(ws + pl.ws_qrows);
  p.part = reinterpret_cast<uint8_t*>(ws + pl.ws_o);
  p.status = status;
  switch (head_dim) {
    case 64: return step_launch_d<64>(p, pl, fmt, stream);
    case 128: return step_launch_d<128>(p, pl, fmt, stream);
    default: return step_launch_d<256>(p, pl, fmt, stream);
  }
}

}  // namespace dfv
