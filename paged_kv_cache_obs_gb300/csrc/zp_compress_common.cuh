// zp_compress_common.cuh — definitions shared by the fused compression pass (zp_compress.cu)
// and its multi-pass form for sequences longer than one cluster (zp_compress_long.cu).
#pragma once

#include <cstdint>
#include <cuda.h>

#include "zp_internal.h"
#include "zp_ptx.cuh"

namespace zp {

constexpr int kThreads = 256;
constexpr int kKeysPerCta = 256;
constexpr int kRows = 128;         // window rows, padded: MMA M of D1 and N of D2
constexpr int kMaxCluster = 16;    // CTAs per cluster: 8 (portable, 2 CTAs per SM) or 16 (1 per SM)
constexpr int kMaxEvict = 32;      // E = L - k = b <= 32
// table entries cached per request for a cluster of up to MAXC CTAs (256 keys each, b >= 16)
constexpr int max_table(int maxc) { return maxc * (kKeysPerCta / 16); }
constexpr uint32_t kTmemCols = 256;
constexpr uint64_t kWaitNs = 2000000000ull;  // 2 s: far above any legitimate wait

struct CompressArgs {
  uint8_t* pool;
  int64_t num_blocks;
  const int32_t* block_tables;
  const int32_t* dst_tables;
  const int32_t* seq_len;
  const int32_t* qslot;
  const int32_t* n_max_req;         // per-request block budgets, or nullptr
  float* gscores;
  int32_t* err;
  int32_t* work;                    // unit counter of the persistent clusters (zeroed per launch)
  const int32_t* req_order;         // requests grouped by length (variable-length form), or nullptr
  const int32_t* bucket;            // (first index into req_order, request count) of this launch
  float* dbg_attn;
  float* dbg_redund;
  float* dbg_score;
  int32_t* dbg_keep;
  int R, layers, Hq, Hkv, d, b, n_max, w, Gq, Rw, L, k, max_blocks, num_qslots;  // L: longest request
  int Lc;                         // key extent of this launch's clusters: min(L, C*256)
  int layer0, nl;                 // the call's layers: [layer0, layer0 + nl) of the `layers`
  float alpha, beta, decay, sl2;  // sl2 = scale * log2(e)
  float inv_rw;                   // 1 / (w * G_q)
  uint32_t block_bytes;           // bytes of one (layer, block): 2 * Hkv * b * d * 2
  uint32_t kv_bytes;              // bytes of the K (or V) part of a block: Hkv * b * d * 2
  uint32_t row_bytes;             // d * 2
  int b_shift;                    // log2(b)
  int protect_window, causal;
  uint64_t stall_ns;              // test hook (multi-pass form only): 0, or the limit of a wait
                                  // that nothing completes, made at the start of the statistics
};

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ float lg2(float x) {
  float y;
  asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Monotone map float -> uint32 (NaN ranks with -inf, -0 with +0).
__device__ __forceinline__ uint32_t order_bits(float s) {
  if (s != s) s = -INFINITY;
  if (s == 0.0f) s = 0.0f;
  uint32_t u = __float_as_uint(s);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Eviction key: smaller = evicted first = lower S, and on equal S the later position.
__device__ __forceinline__ unsigned long long evict_key(float s, int t) {
  return (static_cast<unsigned long long>(order_bits(s)) << 32) | (0xFFFFFFFFu - static_cast<uint32_t>(t));
}

__device__ __forceinline__ void record_error(int32_t* err, int code) {
  if (err) atomicCAS(err, 0, code);
}

// Byte offset of row `row` of block `phys`, relative to this unit's head base (layer, K, head).
__device__ __forceinline__ size_t row_off_bytes(const CompressArgs& a, int phys, int kv, int row) {
  return static_cast<size_t>(static_cast<uint32_t>(phys)) * a.block_bytes + kv * a.kv_bytes +
         static_cast<uint32_t>(row) * a.row_bytes;
}

// Pass 1 of one window row over one 128-column half of a 256-key tile of scores in TMEM (row =
// this thread's TMEM lane, columns from `tl`): the row's max and its exp2-sum relative to that
// max, over the scaled scores (scale sl2) of columns [0, ncol), of which [0, vlim) are visible to
// this row and [0, vall) to every row.  Online over two 64-column chunks: the chunk's max, then
// its exponentials against the running max (the sum so far is rescaled when the max grows);
// two 32-column loads per wait and four partial sums.  A group of 32 columns that every row
// sees whole takes the unpredicated path; the others compare each column with this row's limit.
// A row with no visible column gives (-inf, 0).
__device__ __forceinline__ float2 row_stats_half(uint32_t tl, int ncol, int vlim, int vall, float sl2) {
  float m = -INFINITY;
  float ls[4] = {0.0f, 0.0f, 0.0f, 0.0f};
  for (int c2 = 0; c2 < 2; ++c2) {
    const int col0 = c2 * 64;
    if (col0 >= ncol) break;
    uint32_t ra[32], rb[32];
    tmem_ld32_issue(tl + col0, ra);
    tmem_ld32_issue(tl + col0 + 32, rb);
    tmem_wait_ld(ra);
    tmem_ld_dep(rb);
    const bool fa = col0 + 32 <= vall, fb = col0 + 64 <= vall;  // groups every row sees whole
    const int la = vlim - col0, lb = vlim - col0 - 32;          // visible columns of each group
    float mx[4] = {m, m, m, m};
    if (fa) {
#pragma unroll
      for (int j = 0; j < 32; ++j) mx[j & 3] = fmaxf(mx[j & 3], __uint_as_float(ra[j]));
    } else {
#pragma unroll
      for (int j = 0; j < 32; ++j)
        if (j < la) mx[j & 3] = fmaxf(mx[j & 3], __uint_as_float(ra[j]));
    }
    if (fb) {
#pragma unroll
      for (int j = 0; j < 32; ++j) mx[j & 3] = fmaxf(mx[j & 3], __uint_as_float(rb[j]));
    } else {
#pragma unroll
      for (int j = 0; j < 32; ++j)
        if (j < lb) mx[j & 3] = fmaxf(mx[j & 3], __uint_as_float(rb[j]));
    }
    const float mn = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3]));
    if (mn == -INFINITY) continue;  // nothing visible yet
    if (m != -INFINITY && mn > m) {
      const float corr = ex2((m - mn) * sl2);
#pragma unroll
      for (int e = 0; e < 4; ++e) ls[e] *= corr;
    }
    m = mn;
    const float mo = m * sl2;
    if (fa) {
#pragma unroll
      for (int j = 0; j < 32; ++j) ls[j & 3] += ex2(fmaf(__uint_as_float(ra[j]), sl2, -mo));
    } else {
#pragma unroll
      for (int j = 0; j < 32; ++j)
        if (j < la) ls[j & 3] += ex2(fmaf(__uint_as_float(ra[j]), sl2, -mo));
    }
    if (fb) {
#pragma unroll
      for (int j = 0; j < 32; ++j) ls[j & 3] += ex2(fmaf(__uint_as_float(rb[j]), sl2, -mo));
    } else {
#pragma unroll
      for (int j = 0; j < 32; ++j)
        if (j < lb) ls[j & 3] += ex2(fmaf(__uint_as_float(rb[j]), sl2, -mo));
    }
  }
  return make_float2(m, (ls[0] + ls[1]) + (ls[2] + ls[3]));
}

// Pass 2 for one key over the window rows of a score tile in TMEM (key = this thread's TMEM
// lane, rows as columns from `tl`): the sum over the rows i < Rw that see the key (i >= imin, or
// every row when all_rows) of exp2(s_i * sl2 - row_off[i]), row_off[i] being row i's log2
// normaliser in scaled units (+inf for padding rows, which add 0).  Two 32-column loads per
// wait, four partial sums; row_off is read as float4 (16-byte aligned).
__device__ __forceinline__ float key_mass(uint32_t tl, int Rw, bool all_rows, int imin, const float* row_off,
                                          float sl2) {
  const float4* off4 = reinterpret_cast<const float4*>(row_off);
  float acc[4] = {0.0f, 0.0f, 0.0f, 0.0f};
  for (int c2 = 0; c2 < 2; ++c2) {
    if (c2 * 64 >= Rw) break;
    uint32_t ra[32], rb[32];
    tmem_ld32_issue(tl + c2 * 64, ra);
    tmem_ld32_issue(tl + c2 * 64 + 32, rb);
    tmem_wait_ld(ra);
    tmem_ld_dep(rb);
#pragma unroll
    for (int q = 0; q < 16; ++q) {
      const float4 o = off4[c2 * 16 + q];
      const float oo[4] = {o.x, o.y, o.z, o.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int jj = 4 * q + e;  // 0..63 within this pair of loads
        const float v = __uint_as_float(jj < 32 ? ra[jj & 31] : rb[jj & 31]);
        const float p = ex2(fmaf(v, sl2, -oo[e]));
        if (all_rows || c2 * 64 + jj >= imin) acc[e] += p;
      }
    }
  }
  return (acc[0] + acc[1]) + (acc[2] + acc[3]);
}

// Lightning redundancy of the 32 keys [key0, key0 + 32) of one warp (BW = block size 16 or 32;
// KS = d / 16 k-steps, unrolled, or KS = 0: a loop over the d / 16 k-steps, which keeps fewer
// registers live), from K in 128-byte-swizzled shared memory, with warp-level mma.sync:
// the BW x BW Gram of each block (G = K K^T, so one ldmatrix per k-step gives both the A and the
// B fragments), squared norms from its diagonal, and the in-block row sums of cos(k_t, k_j),
// j != t, over the tokens the block holds (keys at or past L are excluded).  Returns the
// redundancy of key key0 + lane.  The unrolled form takes reciprocal norms by rsqrt (clamped
// like 1 / max(norm, 1e-12)) and divides the mean with the fast reciprocal, both within a few
// ulp of the loop form's IEEE square root and divisions.
template <int BW, int KS>
__device__ __forceinline__ float lightning_redundancy_ks(const uint8_t (&K)[2][kKeysPerCta * 128], float* inv_n,
                                                         int key0, int lane, int d, int t0, int L) {
  constexpr int NT = BW / 8;  // n8 tiles per m16 row tile
  float acc[2][NT][4];
#pragma unroll
  for (int mt = 0; mt < 2; ++mt)
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) acc[mt][nt][e] = 0.0f;
  // The k-steps: with KS > 0 the outer loop is unrolled KS times and the inner one runs once;
  // with KS = 0 the outer one runs once and the inner one loops over d / 16 (the code the
  // compiler generates for that form is the one the register budget of the fused kernel was
  // set with).  A k-step loads both m-tiles' fragments by ldmatrix, then runs the block Gram
  // MMAs.
  const int nks = KS > 0 ? KS : (d >> 4);
#pragma unroll
  for (int ks = 0; ks < (KS > 0 ? KS : 1); ++ks)
    for (int ks2 = ks; ks2 < nks; ks2 += (KS > 0 ? nks : 1)) {
      uint32_t f[2][4];
#pragma unroll
      for (int mt = 0; mt < 2; ++mt) {
        const int row = key0 + 16 * mt + (lane & 7) + ((lane >> 3) & 1) * 8;
        const int chunk = 2 * ks2 + (lane >> 4);
        ldmatrix_x4(smem_u32(&K[chunk >> 3][row * 128 + (((chunk & 7) ^ (row & 7)) << 4)]), f[mt]);
      }
#pragma unroll
      for (int mt = 0; mt < 2; ++mt)
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          // columns 8nt..8nt+7 of the block: rows (sub = nt&1) of m-tile src of the same fragments
          const int src = (BW == 16) ? mt : (nt >> 1);
          const int sub = nt & 1;
          mma_16816_bf16(acc[mt][nt], f[mt], sub ? f[src][1] : f[src][0], sub ? f[src][3] : f[src][2]);
        }
    }
  const int g = lane >> 2, tq = lane & 3;
  // squared norms from the diagonal -> reciprocal norms in shared memory
#pragma unroll
  for (int mt = 0; mt < 2; ++mt)
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int row = 16 * mt + g + 8 * (e >> 1);
        const int col = (BW == 16 ? 16 * mt : 0) + 8 * nt + 2 * tq + (e & 1);
        if (row == col) {
          if constexpr (KS > 0)
            inv_n[key0 + row] = fminf(rsqrtf(fmaxf(acc[mt][nt][e], 0.0f)), 1e12f);
          else
            inv_n[key0 + row] = 1.0f / fmaxf(sqrtf(fmaxf(acc[mt][nt][e], 0.0f)), 1e-12f);
        }
      }
  __syncwarp();
  float rr[2][2];  // redundancy of rows 16mt + 8hf + g
#pragma unroll
  for (int mt = 0; mt < 2; ++mt)
#pragma unroll
    for (int hf = 0; hf < 2; ++hf) {
      const int row = 16 * mt + 8 * hf + g;
      float sum = 0.0f;
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int col = (BW == 16 ? 16 * mt : 0) + 8 * nt + 2 * tq + e;
          const bool ok = col != row && t0 + key0 + col < L;
          sum += ok ? acc[mt][nt][2 * hf + e] * inv_n[key0 + col] : 0.0f;
        }
      sum += __shfl_xor_sync(0xffffffffu, sum, 1);
      sum += __shfl_xor_sync(0xffffffffu, sum, 2);
      const int bstart = (BW == 16) ? 16 * mt : 0;             // block of this row within the warp
      const int m = min(BW, L - (t0 + key0 + bstart));         // tokens the block holds
      if constexpr (KS > 0)
        rr[mt][hf] = m > 1 ? __fdividef(sum * inv_n[key0 + row], static_cast<float>(m - 1)) : 0.0f;
      else
        rr[mt][hf] = m > 1 ? sum * inv_n[key0 + row] / static_cast<float>(m - 1) : 0.0f;
    }
  // deliver: lane k takes row k, computed by lane 4 * (k % 8)
  const int srcl = 4 * (lane & 7);
  const float v00 = __shfl_sync(0xffffffffu, rr[0][0], srcl), v01 = __shfl_sync(0xffffffffu, rr[0][1], srcl);
  const float v10 = __shfl_sync(0xffffffffu, rr[1][0], srcl), v11 = __shfl_sync(0xffffffffu, rr[1][1], srcl);
  const int mt = lane >> 4, hf = (lane >> 3) & 1;
  return mt ? (hf ? v11 : v10) : (hf ? v01 : v00);
}

// Unrolled for d = 128 and d = 64 (twice the code, about half the latency of the loop).
template <int BW>
__device__ __forceinline__ float warp_lightning_redundancy(const uint8_t (&K)[2][kKeysPerCta * 128], float* inv_n,
                                                           int key0, int lane, int d, int t0, int L) {
  return d == 128 ? lightning_redundancy_ks<BW, 8>(K, inv_n, key0, lane, d, t0, L)
                  : lightning_redundancy_ks<BW, 4>(K, inv_n, key0, lane, d, t0, L);
}

// The loop form, for a kernel whose registers are already tight.
template <int BW>
__device__ __forceinline__ float warp_lightning_redundancy_rolled(const uint8_t (&K)[2][kKeysPerCta * 128],
                                                                  float* inv_n, int key0, int lane, int d, int t0,
                                                                  int L) {
  return lightning_redundancy_ks<BW, 0>(K, inv_n, key0, lane, d, t0, L);
}


// Multi-pass compression of sequences longer than one cluster (L > 4096), in
// zp_compress_long.cu.  `scratch` is the workspace past its first 256 bytes.
size_t compress_long_scratch_bytes(int64_t units, int L);
zp_status launch_compress_long(const CUtensorMap& tmK, const CUtensorMap& tmQ, const CompressArgs& a,
                               void* scratch, cudaStream_t st);

}  // namespace zp
