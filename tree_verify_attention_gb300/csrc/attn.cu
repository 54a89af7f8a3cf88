// Tree-masked split-K flash-decode attention over a Q4_0 KV cache.
//
// "Luce DFlash: Qwen3.6-27B ..." (ai-navigate-news, ja), feature list: the
// target verifies the DDTree draft tree (block size 16, budget 22) in one
// forward, with sliding-window flash attention at decode (window 2048) over
// a Q4_0 KV cache. Each tree node attends to the committed keys inside its
// window and to its own ancestors (and itself) in the tree.
//
// Work split. For one KV head, the rows are the (node, query head) pairs
// of its GQA group: R = N * Hq/Hkv (138 at budget 22, 24/4 heads). A CTA
// owns one KV head, one block of up to 128 rows and one contiguous range
// of 64-key tiles; the tile list is the committed keys of the widest
// window (the root's) followed by the tree nodes' own keys. Splits write
// unnormalised partials (O, running max, running sum) that a second small
// kernel merges by log-sum-exp; with one split the kernel writes the
// output directly.
//
// Per tile: the Q4_0 rows of K and V (contiguous per head: 64 keys x 144
// bytes at D = 256) arrive by 1-D bulk copy into a double-buffered raw
// stage, completing on an mbarrier; all threads then dequantise them into
// fp16 tiles ((q - 8) * d, one rounding), and each warp runs 16 rows of
// S = Q K^T, the masked online softmax in registers, and O += P V on the
// tensor cores (mma.sync m16n8k16, f32 accumulate).

#include <math.h>

#include "common.cuh"

namespace dfv {

constexpr int kTile = 64;            // keys per tile
constexpr int kAttnThreads = 256;    // 8 warps; warps beyond rows/16 only stage data
constexpr int kMaxRowsPerCta = 128;
constexpr int kMaxSplits = 256;

struct AttnPlan {
  int rows, n_rb, rb_rows, splits, smem;
};

struct AttnParams {
  int n_nodes, max_depth, hq, hkv, group, window, capacity;
  int rows, n_rb, rb_rows, splits;
  float scale_log2;
  const int32_t* ctx_len;
  const uint8_t* k_cache;
  const uint8_t* v_cache;
  const __nv_bfloat16* q;
  const __nv_bfloat16* tree_k;
  const __nv_bfloat16* tree_v;
  const int32_t* parent;
  float* out;
  float* lse;
  float* part_o;      // [hkv][n_rb][splits][rb_rows][D]
  float2* part_ml;    // [hkv][n_rb][splits][rb_rows]  (running max (log2 units), sum)
  uint32_t* status;
};

template <int D>
struct AttnSmem {
  static constexpr int kRowB = D / 32 * 18;             // bytes of one Q4_0 row
  static constexpr bool kBulk = (kRowB % 16) == 0;      // bulk-copy staging possible
  static constexpr int kLd = D + 8;                     // fp16 row stride (bank spread)
  static constexpr int kTileHalfBytes = kTile * kLd * 2;
  static constexpr int kRawStage = kBulk ? 2 * kTile * kRowB : 0;
  static int bytes(int rb_rows) {
    return rb_rows * kLd * 2 + 2 * kTileHalfBytes + 2 * kRawStage + 16;
  }
};

static int round_up(int x, int m) { return (x + m - 1) / m * m; }

static AttnPlan attn_plan(int n_nodes, int hq, int hkv, int head_dim, int window, int cap) {
  AttnPlan pl;
  pl.rows = n_nodes * (hq / hkv);
  pl.n_rb = (pl.rows + kMaxRowsPerCta - 1) / kMaxRowsPerCta;
  pl.rb_rows = round_up((pl.rows + pl.n_rb - 1) / pl.n_rb, 16);
  const long kbound = window > 0 ? (window - 1 < cap ? window - 1 : cap) : cap;
  const long tiles = (kbound + kTile - 1) / kTile + (n_nodes + kTile - 1) / kTile;
  long s = sm_count() / (hkv * pl.n_rb);
  if (s > tiles) s = tiles;
  if (s > kMaxSplits) s = kMaxSplits;
  if (s < 1) s = 1;
  pl.splits = static_cast<int>(s);
  switch (head_dim) {
    case 64: pl.smem = AttnSmem<64>::bytes(pl.rb_rows); break;
    case 128: pl.smem = AttnSmem<128>::bytes(pl.rb_rows); break;
    default: pl.smem = AttnSmem<256>::bytes(pl.rb_rows); break;
  }
  return pl;
}

static size_t attn_ws_bytes(const AttnPlan& pl, int hkv, int head_dim) {
  if (pl.splits == 1) return 256;
  const size_t n = static_cast<size_t>(hkv) * pl.n_rb * pl.splits * pl.rb_rows;
  return n * head_dim * sizeof(float) + n * sizeof(float2) + 256;
}

template <int D>
__global__ void __launch_bounds__(kAttnThreads, 1) attn_split_kernel(AttnParams p) {
  using L = AttnSmem<D>;
  constexpr int NB = D / 32;
  extern __shared__ __align__(128) uint8_t smem[];
  __half* sQ = reinterpret_cast<__half*>(smem);
  __half* sK = reinterpret_cast<__half*>(smem + p.rb_rows * L::kLd * 2);
  __half* sV = sK + kTile * L::kLd;
  uint8_t* raw = reinterpret_cast<uint8_t*>(sV + kTile * L::kLd);
  uint64_t* bars = reinterpret_cast<uint64_t*>(raw + 2 * L::kRawStage);

  __shared__ int s_J[kMaxNodes], s_dep[kMaxNodes];
  __shared__ uint32_t s_anc[kMaxNodes][kMaskWords];
  __shared__ int s_row_node[kMaxRowsPerCta], s_row_lo[kMaxRowsPerCta];
  __shared__ int s_ok;

  const int split = blockIdx.x, rb = blockIdx.y, h = blockIdx.z;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int N = p.n_nodes, RB = p.rb_rows;
  const bool first_cta = (blockIdx.x | blockIdx.y | blockIdx.z) == 0;

  int C = *p.ctx_len;
  if (C < 0 || C > p.capacity) {
    if (first_cta && tid == 0) report(p.status, DFV_DEV_CTX);
    C = C < 0 ? 0 : p.capacity;
  }
  const int lo_min = p.window > 0 ? max(0, C - p.window + 1) : 0;
  const int nct = (C - lo_min + kTile - 1) / kTile;          // committed tiles
  const int T = nct + (N + kTile - 1) / kTile;               // + tree tiles
  const int t_begin = static_cast<int>(static_cast<long>(split) * T / p.splits);
  const int t_end = static_cast<int>(static_cast<long>(split + 1) * T / p.splits);

  auto issue = [&](int tile, int stage) {
    const int j0 = lo_min + tile * kTile;
    const int nk = min(kTile, C - j0);
    const uint32_t bytes = static_cast<uint32_t>(nk * L::kRowB);
    const size_t off = (static_cast<size_t>(h) * p.capacity + j0) * L::kRowB;
    uint8_t* dst = raw + stage * L::kRawStage;
    fence_proxy_async_smem();
    mbar_arrive_expect_tx(&bars[stage], 2 * bytes);
    bulk_g2s(dst, p.k_cache + off, bytes, &bars[stage]);
    bulk_g2s(dst + kTile * L::kRowB, p.v_cache + off, bytes, &bars[stage]);
  };

  if constexpr (L::kBulk) {
    if (tid == 0) {
      mbar_init(&bars[0], 1);
      mbar_init(&bars[1], 1);
      fence_mbar_init();
      if (t_begin < t_end && t_begin < nct) issue(t_begin, 0);
    }
  }

  // ---- tree: depth and ancestor-or-self masks by pointer jumping
  if (tid < N) {
    int pa = p.parent[tid];
    if (tid == 0) pa = -1;
    else if (pa < 0 || pa >= tid) {
      if (first_cta) report(p.status, DFV_DEV_BAD_TREE);
      pa = 0;
    }
    s_J[tid] = pa;
    s_dep[tid] = tid > 0 ? 1 : 0;
#pragma unroll
    for (int w = 0; w < kMaskWords; ++w) s_anc[tid][w] = (tid >> 5) == w ? (1u << (tid & 31)) : 0u;
  }
  __syncthreads();
#pragma unroll 1
  for (int round = 0; round < 7; ++round) {
    int j = -1, nd = 0, nj = -1;
    uint32_t nm[kMaskWords];
    if (tid < N) {
      j = s_J[tid];
      if (j >= 0) {
        nd = s_dep[tid] + s_dep[j];
        nj = s_J[j];
#pragma unroll
        for (int w = 0; w < kMaskWords; ++w) nm[w] = s_anc[tid][w] | s_anc[j][w];
      }
    }
    __syncthreads();
    if (tid < N && j >= 0) {
      s_dep[tid] = nd;
      s_J[tid] = nj;
#pragma unroll
      for (int w = 0; w < kMaskWords; ++w) s_anc[tid][w] = nm[w];
    }
    __syncthreads();
  }
  if (first_cta && tid < N && s_dep[tid] > p.max_depth) report(p.status, DFV_DEV_DEPTH);

  // ---- rows of this CTA
  if (tid < RB) {
    const int rg = rb * RB + tid;
    if (rg < p.rows) {
      const int node = rg / p.group;
      s_row_node[tid] = node;
      s_row_lo[tid] = p.window > 0 ? C + s_dep[node] - p.window + 1 : 0;
    } else {
      s_row_node[tid] = -1;
      s_row_lo[tid] = 0x7fffffff;
    }
  }
  // ---- Q rows -> fp16 smem
  for (int it = tid; it < RB * (D / 8); it += kAttnThreads) {
    const int lr = it / (D / 8), c8 = it % (D / 8);
    const int rg = rb * RB + lr;
    uint4 outv = make_uint4(0, 0, 0, 0);
    if (rg < p.rows) {
      const int node = rg / p.group, qh = h * p.group + rg % p.group;
      const uint4 v = *reinterpret_cast<const uint4*>(
          p.q + (static_cast<size_t>(node) * p.hq + qh) * D + c8 * 8);
      const __nv_bfloat162* b = reinterpret_cast<const __nv_bfloat162*>(&v);
      uint32_t* o = reinterpret_cast<uint32_t*>(&outv);
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float2 f = __bfloat1622float2(b[e]);
        o[e] = pack_half2(f.x, f.y);
      }
    }
    *reinterpret_cast<uint4*>(sQ + lr * L::kLd + c8 * 8) = outv;
  }
  __syncthreads();

  // ---- per-warp state: 16 rows, D/8 output n8-tiles
  const bool mma_warp = warp < RB / 16;
  const int r0 = warp * 16 + (lane >> 2), r1 = r0 + 8;
  int node0 = -1, node1 = -1, lo0 = 0, lo1 = 0;
  if (mma_warp) {
    node0 = s_row_node[r0];
    node1 = s_row_node[r1];
    lo0 = s_row_lo[r0];
    lo1 = s_row_lo[r1];
  }
  float o[D / 8][4];
#pragma unroll
  for (int i = 0; i < D / 8; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
  float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
  uint32_t phase = 0;   // bit s = parity of the next wait on bars[s]

#pragma unroll 1
  for (int tile = t_begin; tile < t_end; ++tile) {
    const int li = tile - t_begin, stage = li & 1;
    const bool committed = tile < nct;
    if constexpr (L::kBulk) {
      if (tid == 0) {
        if (tile + 1 < t_end && tile + 1 < nct) issue(tile + 1, stage ^ 1);
        if (committed) {
          const bool ok = mbar_wait_bounded(&bars[stage], (phase >> stage) & 1u);
          s_ok = ok ? 1 : 0;
        } else {
          s_ok = 1;
        }
      }
      if (committed) phase ^= (1u << stage);
    } else {
      if (tid == 0) s_ok = 1;
    }
    __syncthreads();
    if (!s_ok) {
      if (tid == 0) report(p.status, DFV_DEV_TIMEOUT);
      return;
    }
    // ---- dequantise / convert the tile into sK, sV (fp16)
    if (committed) {
      const int j0 = lo_min + tile * kTile;
      const int nk = min(kTile, C - j0);
      for (int it = tid; it < 2 * kTile * NB; it += kAttnThreads) {
        const int kv = it / (kTile * NB);
        const int key = (it / NB) % kTile;
        const int b = it % NB;
        __half* dst = (kv ? sV : sK) + key * L::kLd + b * 32;
        if (key < nk) {
          const uint8_t* blk;
          if constexpr (L::kBulk) {
            blk = raw + stage * L::kRawStage + kv * kTile * L::kRowB + key * L::kRowB + b * 18;
          } else {
            blk = (kv ? p.v_cache : p.k_cache) +
                  (static_cast<size_t>(h) * p.capacity + j0 + key) * L::kRowB + b * 18;
          }
          const uint16_t* w = reinterpret_cast<const uint16_t*>(blk);
          q4_0_block_to_half(w + 1, __ushort_as_half(w[0]), dst, dst + 16);
        } else {
#pragma unroll
          for (int e = 0; e < 32; e += 8)
            *reinterpret_cast<uint4*>(dst + e) = make_uint4(0, 0, 0, 0);
        }
      }
    } else {
      const int t0 = (tile - nct) * kTile;
      for (int it = tid; it < 2 * kTile * (D / 8); it += kAttnThreads) {
        const int kv = it / (kTile * (D / 8));
        const int key = (it / (D / 8)) % kTile;
        const int c8 = it % (D / 8);
        uint4 outv = make_uint4(0, 0, 0, 0);
        const int t = t0 + key;
        if (t < N) {
          const __nv_bfloat16* src = (kv ? p.tree_v : p.tree_k) +
                                     (static_cast<size_t>(t) * p.hkv + h) * D + c8 * 8;
          const uint4 v = *reinterpret_cast<const uint4*>(src);
          const __nv_bfloat162* b = reinterpret_cast<const __nv_bfloat162*>(&v);
          uint32_t* ov = reinterpret_cast<uint32_t*>(&outv);
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float2 f = __bfloat1622float2(b[e]);
            ov[e] = pack_half2(f.x, f.y);
          }
        }
        *reinterpret_cast<uint4*>((kv ? sV : sK) + key * L::kLd + c8 * 8) = outv;
      }
    }
    __syncthreads();

    if (mma_warp) {
      // ---- S = Q K^T for 16 rows x 64 keys
      float s[8][4];
#pragma unroll
      for (int i = 0; i < 8; ++i) s[i][0] = s[i][1] = s[i][2] = s[i][3] = 0.f;
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        uint32_t a0, a1, a2, a3;
        ldsm_x4(a0, a1, a2, a3, sQ + (warp * 16 + (lane & 15)) * L::kLd + kk * 16 + (lane >> 4) * 8);
#pragma unroll
        for (int np = 0; np < 4; ++np) {
          uint32_t b0, b1, b2, b3;
          ldsm_x4(b0, b1, b2, b3,
                  sK + (np * 16 + (lane >> 4) * 8 + (lane & 7)) * L::kLd + kk * 16 +
                      ((lane >> 3) & 1) * 8);
          mma_f16(s[2 * np], a0, a1, a2, a3, b0, b1);
          mma_f16(s[2 * np + 1], a0, a1, a2, a3, b2, b3);
        }
      }
      // ---- scale, mask, online softmax (base 2)
      float mx0 = -INFINITY, mx1 = -INFINITY;
      if (committed) {
        const int j0 = lo_min + tile * kTile;
        const int nk = min(kTile, C - j0);
#pragma unroll
        for (int nt = 0; nt < 8; ++nt)
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int key = nt * 8 + (lane & 3) * 2 + (e & 1);
            const int lo = e < 2 ? lo0 : lo1;
            const bool vis = key < nk && j0 + key >= lo;
            s[nt][e] = vis ? s[nt][e] * p.scale_log2 : -INFINITY;
          }
      } else {
        const int t0 = (tile - nct) * kTile;
#pragma unroll
        for (int nt = 0; nt < 8; ++nt)
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int t = t0 + nt * 8 + (lane & 3) * 2 + (e & 1);
            const int node = e < 2 ? node0 : node1;
            const bool vis = node >= 0 && t < N && ((s_anc[node][t >> 5] >> (t & 31)) & 1u);
            s[nt][e] = vis ? s[nt][e] * p.scale_log2 : -INFINITY;
          }
      }
#pragma unroll
      for (int nt = 0; nt < 8; ++nt) {
        mx0 = fmaxf(mx0, fmaxf(s[nt][0], s[nt][1]));
        mx1 = fmaxf(mx1, fmaxf(s[nt][2], s[nt][3]));
      }
      mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
      mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
      mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
      mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
      const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
      const float sub0 = mn0 == -INFINITY ? 0.f : mn0;
      const float sub1 = mn1 == -INFINITY ? 0.f : mn1;
      const float al0 = exp2f(m0 - sub0), al1 = exp2f(m1 - sub1);
      float rs0 = 0.f, rs1 = 0.f;
#pragma unroll
      for (int nt = 0; nt < 8; ++nt) {
        s[nt][0] = exp2f(s[nt][0] - sub0);
        s[nt][1] = exp2f(s[nt][1] - sub0);
        s[nt][2] = exp2f(s[nt][2] - sub1);
        s[nt][3] = exp2f(s[nt][3] - sub1);
        rs0 += s[nt][0] + s[nt][1];
        rs1 += s[nt][2] + s[nt][3];
      }
      l0 = l0 * al0 + rs0;
      l1 = l1 * al1 + rs1;
      m0 = mn0;
      m1 = mn1;
#pragma unroll
      for (int i = 0; i < D / 8; ++i) {
        o[i][0] *= al0;
        o[i][1] *= al0;
        o[i][2] *= al1;
        o[i][3] *= al1;
      }
      // ---- O += P V
#pragma unroll
      for (int kk = 0; kk < kTile / 16; ++kk) {
        const uint32_t a0 = pack_half2(s[2 * kk][0], s[2 * kk][1]);
        const uint32_t a1 = pack_half2(s[2 * kk][2], s[2 * kk][3]);
        const uint32_t a2 = pack_half2(s[2 * kk + 1][0], s[2 * kk + 1][1]);
        const uint32_t a3 = pack_half2(s[2 * kk + 1][2], s[2 * kk + 1][3]);
#pragma unroll
        for (int dp = 0; dp < D / 16; ++dp) {
          uint32_t b0, b1, b2, b3;
          ldsm_x4_t(b0, b1, b2, b3,
                    sV + (kk * 16 + ((lane >> 3) & 1) * 8 + (lane & 7)) * L::kLd + dp * 16 +
                        (lane >> 4) * 8);
          mma_f16(o[2 * dp], a0, a1, a2, a3, b0, b1);
          mma_f16(o[2 * dp + 1], a0, a1, a2, a3, b2, b3);
        }
      }
    }
    __syncthreads();   // sK / sV are rewritten by the next tile
  }

  if (!mma_warp) return;
  l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
  l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
  l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
  l1 += __shfl_xor_sync(0xffffffffu, l1, 2);

  const int col = (lane & 3) * 2;
#pragma unroll
  for (int half = 0; half < 2; ++half) {
    const int lr = half ? r1 : r0;
    const int rg = rb * RB + lr;
    if (rg >= p.rows) continue;
    const float m = half ? m1 : m0, l = half ? l1 : l0;
    if (p.splits == 1) {
      const int node = rg / p.group, qh = h * p.group + rg % p.group;
      float* dst = p.out + (static_cast<size_t>(node) * p.hq + qh) * D;
      const float inv = 1.f / l;
#pragma unroll
      for (int i = 0; i < D / 8; ++i)
        *reinterpret_cast<float2*>(dst + i * 8 + col) =
            make_float2(o[i][2 * half] * inv, o[i][2 * half + 1] * inv);
      if (p.lse != nullptr && (lane & 3) == 0)
        p.lse[node * p.hq + qh] = (m + log2f(l)) * 0.69314718055994531f;
    } else {
      const size_t prow =
          ((static_cast<size_t>(h) * p.n_rb + rb) * p.splits + split) * RB + lr;
      float* dst = p.part_o + prow * D;
#pragma unroll
      for (int i = 0; i < D / 8; ++i)
        *reinterpret_cast<float2*>(dst + i * 8 + col) =
            make_float2(o[i][2 * half], o[i][2 * half + 1]);
      if ((lane & 3) == 0) p.part_ml[prow] = make_float2(m, l);
    }
  }
}

// Merge split partials of one (KV head, row) by log-sum-exp.
constexpr int kCombineThreads = 64;

template <int D>
__global__ void __launch_bounds__(kCombineThreads) attn_combine_kernel(AttnParams p) {
  __shared__ float s_w[kMaxSplits];
  __shared__ float s_M, s_l;
  const int h = blockIdx.y, rg = blockIdx.x;
  const int rb = rg / p.rb_rows, lr = rg % p.rb_rows;
  const size_t base = (static_cast<size_t>(h) * p.n_rb + rb) * p.splits;
  if (threadIdx.x < 32) {
    float M = -INFINITY;
    for (int s = threadIdx.x; s < p.splits; s += 32)
      M = fmaxf(M, p.part_ml[(base + s) * p.rb_rows + lr].x);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
    float l = 0.f;
    for (int s = threadIdx.x; s < p.splits; s += 32) {
      const float2 ml = p.part_ml[(base + s) * p.rb_rows + lr];
      const float w = ml.x == -INFINITY ? 0.f : exp2f(ml.x - M);
      s_w[s] = w;
      l += w * ml.y;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) l += __shfl_xor_sync(0xffffffffu, l, o);
    if (threadIdx.x == 0) {
      s_M = M;
      s_l = l;
    }
  }
  __syncthreads();
  const float inv = 1.f / s_l;
  const int node = rg / p.group, qh = h * p.group + rg % p.group;
  for (int d = threadIdx.x * 4; d < D; d += kCombineThreads * 4) {
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int s = 0; s < p.splits; ++s) {
      const float w = s_w[s];
      if (w == 0.f) continue;
      const float4 v = *reinterpret_cast<const float4*>(
          p.part_o + ((base + s) * p.rb_rows + lr) * static_cast<size_t>(D) + d);
      acc.x += w * v.x;
      acc.y += w * v.y;
      acc.z += w * v.z;
      acc.w += w * v.w;
    }
    *reinterpret_cast<float4*>(p.out + (static_cast<size_t>(node) * p.hq + qh) * D + d) =
        make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
  }
  if (threadIdx.x == 0 && p.lse != nullptr)
    p.lse[node * p.hq + qh] = (s_M + log2f(s_l)) * 0.69314718055994531f;
}

template <int D>
static dfv_status attn_launch_d(const AttnParams& p, const AttnPlan& pl, cudaStream_t stream) {
  static int configured_smem[64] = {};   // per device ordinal
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return DFV_ERR_CUDA;
  if (configured_smem[dev] < pl.smem) {
    if (cudaFuncSetAttribute(attn_split_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             pl.smem) != cudaSuccess)
      return DFV_ERR_CUDA;
    configured_smem[dev] = pl.smem;
  }
  dim3 grid(pl.splits, pl.n_rb, p.hkv);
  attn_split_kernel<D><<<grid, kAttnThreads, pl.smem, stream>>>(p);
  if (cudaGetLastError() != cudaSuccess) return DFV_ERR_CUDA;
  if (pl.splits > 1) {
    attn_combine_kernel<D><<<dim3(pl.rows, p.hkv), kCombineThreads, 0, stream>>>(p);
    if (cudaGetLastError() != cudaSuccess) return DFV_ERR_CUDA;
  }
  return DFV_OK;
}

static bool attn_shape_ok(int n_nodes, int hq, int hkv, int head_dim, int window, int cap) {
  return n_nodes >= 1 && n_nodes <= kMaxNodes && hkv >= 1 && hq >= hkv && hq % hkv == 0 &&
         hq <= 256 && window >= 0 && cap >= 0;
}

size_t attn_workspace_bytes(int n_nodes, int hq, int hkv, int head_dim, int window, int cap) {
  if (!attn_shape_ok(n_nodes, hq, hkv, head_dim, window, cap)) return 0;
  if (head_dim != 64 && head_dim != 128 && head_dim != 256) return 0;
  return attn_ws_bytes(attn_plan(n_nodes, hq, hkv, head_dim, window, cap), hkv, head_dim);
}

int attn_launches(int n_nodes, int hq, int hkv, int head_dim, int window, int cap) {
  if (!attn_shape_ok(n_nodes, hq, hkv, head_dim, window, cap)) return -1;
  if (head_dim != 64 && head_dim != 128 && head_dim != 256) return -1;
  return attn_plan(n_nodes, hq, hkv, head_dim, window, cap).splits > 1 ? 2 : 1;
}

dfv_status attn_launch(int n_nodes, int max_depth, int hq, int hkv, int head_dim, int window,
                       int kv_format, int cap, const int32_t* ctx_len, const void* k_cache,
                       const void* v_cache, const void* q, const void* tree_k,
                       const void* tree_v, const int32_t* parent, float scale, float* out,
                       float* lse, void* workspace, size_t ws_bytes, uint32_t* status,
                       cudaStream_t stream) {
  if (!attn_shape_ok(n_nodes, hq, hkv, head_dim, window, cap)) return DFV_ERR_INVALID;
  if (kv_format != DFV_KV_Q4_0) return DFV_ERR_UNSUPPORTED;
  if (head_dim != 64 && head_dim != 128 && head_dim != 256) return DFV_ERR_UNSUPPORTED;
  if (!ctx_len || !k_cache || !v_cache || !q || !tree_k || !tree_v || !parent || !out ||
      !workspace)
    return DFV_ERR_INVALID;
  if (!aligned(k_cache, 16) || !aligned(v_cache, 16) || !aligned(q, 16) || !aligned(tree_k, 16) ||
      !aligned(tree_v, 16) || !aligned(out, 16) || !aligned(workspace, 256))
    return DFV_ERR_INVALID;
  const AttnPlan pl = attn_plan(n_nodes, hq, hkv, head_dim, window, cap);
  if (ws_bytes < attn_ws_bytes(pl, hkv, head_dim)) return DFV_ERR_WORKSPACE;
  AttnParams p;
  p.n_nodes = n_nodes;
  p.max_depth = max_depth;
  p.hq = hq;
  p.hkv = hkv;
  p.group = hq / hkv;
  p.window = window;
  p.capacity = cap;
  p.rows = pl.rows;
  p.n_rb = pl.n_rb;
  p.rb_rows = pl.rb_rows;
  p.splits = pl.splits;
  const float sc = scale > 0.f ? scale : 1.0f / sqrtf(static_cast<float>(head_dim));
  p.scale_log2 = sc * 1.4426950408889634f;
  p.ctx_len = ctx_len;
  p.k_cache = static_cast<const uint8_t*>(k_cache);
  p.v_cache = static_cast<const uint8_t*>(v_cache);
  p.q = static_cast<const __nv_bfloat16*>(q);
  p.tree_k = static_cast<const __nv_bfloat16*>(tree_k);
  p.tree_v = static_cast<const __nv_bfloat16*>(tree_v);
  p.parent = parent;
  p.out = out;
  p.lse = lse;
  const size_t n = static_cast<size_t>(hkv) * pl.n_rb * pl.splits * pl.rb_rows;
  p.part_o = static_cast<float*>(workspace);
  p.part_ml = reinterpret_cast<float2*>(static_cast<char*>(workspace) + n * head_dim * sizeof(float));
  p.status = status;
  switch (head_dim) {
    case 64: return attn_launch_d<64>(p, pl, stream);
    case 128: return attn_launch_d<128>(p, pl, stream);
    default: return attn_launch_d<256>(p, pl, stream);
  }
}

}  // namespace dfv

extern "C" size_t dfv_tree_verify_attn_workspace_bytes(int n_nodes, int n_q_heads, int n_kv_heads,
                                                       int head_dim, int window,
                                                       int cache_capacity) {
  return dfv::attn_workspace_bytes(n_nodes, n_q_heads, n_kv_heads, head_dim, window,
                                   cache_capacity);
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
  return dfv::attn_launch(n_nodes, max_depth, n_q_heads, n_kv_heads, head_dim, window,
                          kv_format, cache_capacity, ctx_len, k_cache, v_cache, q, tree_k,
                          tree_v, parent, scale, out, lse, workspace, workspace_bytes, status,
                          static_cast<cudaStream_t>(stream));
}
