// zp_redundancy.cu — the original all-pairs redundancy score for sm_103a, kept as the ablation of
// the Lightning Redundancy Score.
//
// Operation (Zipage summaries on gist.science: zh §2.1 and es §2 give the O(N^2 b^2) cost of the
// original score over N blocks of b tokens, which Lightning cuts to O(N b^2) by comparing keys
// inside one block only; de §2 notes that the original needs the full similarity matrix).  Per
// unit u = (request r, layer l, kv head h) with L cached tokens:
//   R_all[t] = (1 / (L-1)) * sum_{j < L, j != t} cos(k_t, k_j),   cos with norms clamped at 1e-12,
// and 0 for L < 2 and for t >= L (up to the row length of the output).
//
// GB300 mapping.  One CTA per (unit, 128-row tile of t), 128 threads.  The CTA TMA-loads its 128
// key rows once (A, 128-byte swizzle, one 3-D box per (block, 64-column half)) and streams the
// unit's key tiles (B) through a two-stage ring.  tcgen05 MMA computes each 128 x 128 Gram tile
// A B^T into one of two TMEM accumulators while the four warps reduce the previous one: thread =
// row t (TMEM lane) adds Gram[t][j] / |k_j| over the tile's 128 columns.  The similarity matrix
// is never stored.  R_all[t] = (acc / |k_t| - cos(k_t, k_t)) / (L-1).  All waits are bounded.
#include <algorithm>
#include <mutex>

#include "zp_internal.h"
#include "zp_ptx.cuh"

namespace zp {
namespace {

constexpr int kTile = 128;        // rows per tile = TMEM lanes = MMA M and N
constexpr int kThreadsA = 128;    // thread = row of the CTA's tile
constexpr uint32_t kColsA = 256;  // two 128-column fp32 accumulators
constexpr int kMaxTabA = 256;     // block-table entries per request (L <= 4096 at b = 16)
constexpr uint64_t kWaitNsA = 2000000000ull;

struct ApArgs {
  const uint8_t* pool;
  int32_t num_blocks;
  const int32_t* block_tables;
  const int32_t* seq_len;
  float* out;
  float* sq;                      // [units][L] squared key norms (workspace), from the pre-pass
  int32_t* err;
  int layers, Hkv, d, b, b_shift, max_blocks, L, nt;  // L: launch length, nt: row tiles per unit
};

struct __align__(1024) ApSmem {
  uint8_t A[2][kTile * 128];     // [d-half][row][128 B], 128-byte swizzle: this CTA's rows
  uint8_t B[2][2][kTile * 128];  // [stage][d-half][row][128 B]: the streamed key tiles
  float inv_b[2][kTile];         // reciprocal norms of each stage's rows
  int tab[kMaxTabA];
  uint64_t bar_a, bar_b[2], bar_mma[2];
  uint32_t tmem_base;
};

__device__ __forceinline__ void ap_record_error(int32_t* err, int code) {
  if (err) atomicCAS(err, 0, code);
}

// Zeroes row `row` of a swizzled tile (rows past the sequence must not contribute).
__device__ __forceinline__ void zero_row(uint8_t (&T)[2][kTile * 128], int row, int nhalf) {
  for (int hd = 0; hd < nhalf; ++hd)
#pragma unroll
    for (int ch = 0; ch < 8; ++ch) *reinterpret_cast<uint4*>(&T[hd][row * 128 + ch * 16]) = make_uint4(0, 0, 0, 0);
}

// Issues the TMA of key tile `tile` (rows [128*tile, 128*tile + 128) of the unit) into `dst`,
// only for blocks that hold tokens of the sequence; returns the bytes registered on `bar`.
__device__ __forceinline__ void load_tile(uint8_t (&dst)[2][kTile * 128], const CUtensorMap* tm, uint64_t* bar,
                                          const ApArgs& a, const int* tab, int layer, int h, int tile, int L) {
  const int nhalf = a.d / 64;
  const int blk0 = (tile * kTile) >> a.b_shift;
  const int nblk = min(kTile >> a.b_shift, ((L + a.b - 1) >> a.b_shift) - blk0);
  mbar_arrive_expect_tx(bar, static_cast<uint32_t>(nblk * a.b * a.d * 2));
  for (int bi = 0; bi < nblk; ++bi)
    for (int hd = 0; hd < nhalf; ++hd)
      tma_load_3d(&dst[hd][bi * a.b * 128], tm, bar, hd * 64, h * a.b, layer * a.num_blocks + tab[blk0 + bi]);
}

// Pre-pass: the squared norm of every key of every unit (t < L; 0 past it), in fp32, read once
// from the pool through the block table.  Grid (unit, 128-row tile), thread = key.
__global__ void __launch_bounds__(kThreadsA) key_sq_norm_kernel(const ApArgs a) {
  const int tid = threadIdx.x;
  const int unit = static_cast<int>(blockIdx.x) / a.nt, it = static_cast<int>(blockIdx.x) % a.nt;
  const int h = unit % a.Hkv, layer = (unit / a.Hkv) % a.layers, r = unit / a.Hkv / a.layers;
  const int t = it * kTile + tid;
  if (t >= a.L) return;
  const int L = a.seq_len[r];
  float acc = 0.0f;
  if (L >= 0 && L <= a.L && t < L) {
    const int phys = a.block_tables[static_cast<int64_t>(r) * a.max_blocks + (t >> a.b_shift)];
    if (phys >= 0 && phys < a.num_blocks) {  // bad ids are reported by the main kernel
      const uint4* row = reinterpret_cast<const uint4*>(
          a.pool + ((static_cast<int64_t>(layer) * a.num_blocks + phys) * 2 * a.Hkv + h) * static_cast<int64_t>(a.b) * a.d * 2 +
          static_cast<int64_t>(t & (a.b - 1)) * a.d * 2);
      for (int i = 0; i < a.d / 8; ++i) {
        const uint4 v = row[i];
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float lo = __uint_as_float(w[e] << 16), hi = __uint_as_float(w[e] & 0xFFFF0000u);
          acc = fmaf(lo, lo, acc);
          acc = fmaf(hi, hi, acc);
        }
      }
    }
  }
  a.sq[static_cast<int64_t>(unit) * a.L + t] = acc;
}

__global__ void __launch_bounds__(kThreadsA, 2)
    all_pairs_redundancy_kernel(const __grid_constant__ CUtensorMap tmK, const ApArgs a) {
  extern __shared__ uint8_t smem_raw[];
  ApSmem& s = *reinterpret_cast<ApSmem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int tid = threadIdx.x, warp = tid >> 5;
  const int unit = static_cast<int>(blockIdx.x) / a.nt, it = static_cast<int>(blockIdx.x) % a.nt;
  const int h = unit % a.Hkv, layer = (unit / a.Hkv) % a.layers, r = unit / a.Hkv / a.layers;
  const int nhalf = a.d / 64;
  const int t = it * kTile + tid;  // this thread's row
  float* const out = a.out + static_cast<int64_t>(unit) * a.L;
  const int L = a.seq_len[r];
  if (L < 0 || L > a.L) {
    if (tid == 0 && it == 0) ap_record_error(a.err, ZP_ERR_BAD_TABLE);
    return;
  }
  // rows of this tile past the sequence (or all of them) are 0
  if (t < a.L && (t >= L || L < 2)) out[t] = 0.0f;
  if (it * kTile >= L || L < 2) return;

  const int nblk = (L + a.b - 1) >> a.b_shift;
  bool bad = false;
  for (int i = tid; i < nblk; i += kThreadsA) {
    const int e = a.block_tables[static_cast<int64_t>(r) * a.max_blocks + i];
    s.tab[i] = e;
    bad |= (e < 0 || e >= a.num_blocks);
  }
  if (tid == 0) {
    mbar_init(&s.bar_a, 1);
    mbar_init(&s.bar_b[0], 1);
    mbar_init(&s.bar_b[1], 1);
    mbar_init(&s.bar_mma[0], 1);
    mbar_init(&s.bar_mma[1], 1);
    fence_mbar_init();
    prefetch_tensormap(&tmK);
  }
  if (__syncthreads_or(bad)) {
    if (tid == 0) ap_record_error(a.err, ZP_ERR_BAD_TABLE);
    return;
  }
  if (warp == 0) tmem_alloc(&s.tmem_base, kColsA);
  const int ntc = (L + kTile - 1) / kTile;  // key tiles of the unit
  // (tid 0) mbarrier phases and copies/MMAs in flight, one bit each: bit st for bar_b[st],
  // bit 2 + u for bar_mma[u], bit 4 for bar_a
  uint32_t ph = 0, pend = 0;
  bool ok = true;  // (tid 0)
  if (tid == 0) {
    load_tile(s.A, &tmK, &s.bar_a, a, s.tab, layer, h, it, L);
    pend |= 16u;
    for (int st = 0; st < 2 && st < ntc; ++st) {
      load_tile(s.B[st], &tmK, &s.bar_b[st], a, s.tab, layer, h, st, L);
      pend |= 1u << st;
    }
    ok = mbar_wait_bounded(&s.bar_a, 0, kWaitNsA);
    if (ok) pend &= ~16u;
  }
  tc_fence_before();
  bool fail = __syncthreads_or(!ok);
  tc_fence_after();
  const uint32_t tbase = s.tmem_base;
  float inv_a = 0.0f, self = 0.0f;
  const float* const sq_unit = a.sq + static_cast<int64_t>(unit) * a.L;
  if (!fail) {
    if (t >= L) zero_row(s.A, tid, nhalf);
    const float sq = t < L ? sq_unit[t] : 0.0f;
    inv_a = 1.0f / fmaxf(sqrtf(sq), 1e-12f);
    self = sq * inv_a * inv_a;  // cos(k_t, k_t): 1, or 0 for a zero key
  }
  fence_proxy_async_smem();
  float acc[4] = {0.0f, 0.0f, 0.0f, 0.0f};
  const uint32_t idesc = idesc_bf16_f32(kTile, kTile);
  const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;

  // Reduces the accumulator of key tile j into acc (thread = row).
  auto epilogue = [&](int j) {
    const int u = j & 1;
    if (tid == 0) {
      const bool w = mbar_wait_bounded(&s.bar_mma[u], (ph >> (2 + u)) & 1u, kWaitNsA);
      if (w) {
        ph ^= 4u << u;
        pend &= ~(4u << u);
      }
      ok = ok && w;
    }
    tc_fence_before();
    fail |= __syncthreads_or(!ok);
    tc_fence_after();
    if (fail) return;
#pragma unroll 1
    for (int c4 = 0; c4 < 4; ++c4) {
      uint32_t v[32];
      tmem_ld32_issue(tbase + lane_base + u * kTile + c4 * 32, v);
      tmem_wait_ld(v);
      const float4* ib = reinterpret_cast<const float4*>(&s.inv_b[u][c4 * 32]);
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        const float4 w = ib[q];
        acc[0] = fmaf(__uint_as_float(v[4 * q + 0]), w.x, acc[0]);
        acc[1] = fmaf(__uint_as_float(v[4 * q + 1]), w.y, acc[1]);
        acc[2] = fmaf(__uint_as_float(v[4 * q + 2]), w.z, acc[2]);
        acc[3] = fmaf(__uint_as_float(v[4 * q + 3]), w.w, acc[3]);
      }
    }
  };

  for (int jt = 0; jt < ntc && !fail; ++jt) {
    const int st = jt & 1;
    if (tid == 0) {
      const bool w = mbar_wait_bounded(&s.bar_b[st], (ph >> st) & 1u, kWaitNsA);
      if (w) {
        ph ^= 1u << st;
        pend &= ~(1u << st);
      }
      ok = ok && w;
    }
    fail |= __syncthreads_or(!ok);
    if (fail) break;
    const int tj = jt * kTile + tid;  // the key row this thread normalises
    if (tj >= L) zero_row(s.B[st], tid, nhalf);
    s.inv_b[st][tid] = tj < L ? 1.0f / fmaxf(sqrtf(sq_unit[tj]), 1e-12f) : 0.0f;
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (tid == 0) {
      for (int kk = 0; kk < a.d / 16; ++kk) {
        const uint64_t ad = smem_desc_sw128(smem_u32(&s.A[kk >> 2][(kk & 3) * 32]));
        const uint64_t bd = smem_desc_sw128(smem_u32(&s.B[st][kk >> 2][(kk & 3) * 32]));
        mma_bf16(tbase + st * kTile, ad, bd, idesc, kk > 0);
      }
      mma_commit(&s.bar_mma[st]);
      pend |= 4u << st;
    }
    if (jt >= 1) {
      epilogue(jt - 1);
      if (fail) break;
      // stage (jt + 1) & 1 == (jt - 1) & 1 is free: its MMA has completed and its norms are read
      __syncthreads();
      if (tid == 0 && jt + 1 < ntc) {
        load_tile(s.B[(jt + 1) & 1], &tmK, &s.bar_b[(jt + 1) & 1], a, s.tab, layer, h, jt + 1, L);
        pend |= 1u << ((jt + 1) & 1);
      }
    }
  }
  if (!fail) epilogue(ntc - 1);
  if (!fail && t < L) {
    const float sum = (acc[0] + acc[1]) + (acc[2] + acc[3]);
    out[t] = (sum * inv_a - self) / static_cast<float>(L - 1);
  }
  if (fail && tid == 0) ap_record_error(a.err, ZP_ERR_TIMEOUT);
  // copies and MMAs still in flight after a failed wait: wait for them (bounded) before the
  // shared memory and TMEM are released
  if (tid == 0) {
    if (pend & 16u) mbar_wait_bounded(&s.bar_a, 0, kWaitNsA);
    for (int st = 0; st < 2; ++st) {
      if (pend & (1u << st)) mbar_wait_bounded(&s.bar_b[st], (ph >> st) & 1u, kWaitNsA);
      if (pend & (4u << st)) mbar_wait_bounded(&s.bar_mma[st], (ph >> (2 + st)) & 1u, kWaitNsA);
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0) tmem_dealloc(tbase, kColsA);
}

// two CTAs per SM (228 KB of shared memory per SM, 1 KB reserved per CTA, 1 KB alignment slack)
static_assert(sizeof(ApSmem) + 1024 <= (228 * 1024 - 2 * 1024) / 2, "shared memory must allow two CTAs per SM");

}  // namespace
}  // namespace zp

using namespace zp;

extern "C" size_t zp_redundancy_workspace_size(const zp_params* p, int32_t num_requests, int32_t max_seq_len) {
  if (!p || num_requests < 0) return 0;
  const int64_t L = max_seq_len > 0 ? max_seq_len : static_cast<int64_t>(p->n_max) * p->block_size;
  // error word, then the squared key norms of every unit
  return 256 + static_cast<size_t>(num_requests) * p->num_layers * p->num_kv_heads * static_cast<size_t>(L) * 4;
}

extern "C" zp_status zp_redundancy_all_pairs(const zp_kv_pool* pool, const int32_t* block_tables,
                                             const zp_seq_meta* meta, const zp_params* p, float* redund,
                                             void* workspace, size_t workspace_bytes, zp_stream stream) {
  zp::NvtxRange nvtx_range("zp_redundancy_all_pairs");
  if (!pool || !meta || !p || !workspace) return ZP_ERR_INVALID_ARG;
  if (!pool->base || pool->num_blocks <= 0) return ZP_ERR_INVALID_ARG;
  const int R = meta->num_requests;
  if (R < 0) return ZP_ERR_INVALID_ARG;
  if (R > 0 && (!block_tables || !meta->seq_len || !redund)) return ZP_ERR_INVALID_ARG;
  if (workspace_bytes < zp_redundancy_workspace_size(p, R, meta->max_seq_len) || !aligned(workspace, 256))
    return ZP_ERR_INVALID_ARG;
  const int layers = p->num_layers, Hkv = p->num_kv_heads, d = p->head_dim, b = p->block_size;
  if (layers <= 0 || Hkv <= 0 || p->n_max < 1) return ZP_ERR_INVALID_ARG;
  const int L = meta->max_seq_len > 0 ? meta->max_seq_len : p->n_max * b;
  if (d != 64 && d != 128) return ZP_ERR_UNSUPPORTED;
  if (b != 16 && b != 32) return ZP_ERR_UNSUPPORTED;
  if (L < 1 || (L + b - 1) / b > kMaxTabA || L > kMaxTabA * 16) return ZP_ERR_UNSUPPORTED;
  if (meta->max_blocks < (L + b - 1) / b) return ZP_ERR_INVALID_ARG;
  if (!aligned(pool->base, 16)) return ZP_ERR_INVALID_ARG;
  if (static_cast<int64_t>(layers) * pool->num_blocks >= (int64_t(1) << 31)) return ZP_ERR_UNSUPPORTED;
  const int nt = (L + kTile - 1) / kTile;
  const int64_t ctas = static_cast<int64_t>(R) * layers * Hkv * nt;
  if (ctas >= (int64_t(1) << 31)) return ZP_ERR_UNSUPPORTED;

  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (cudaMemsetAsync(workspace, 0, 4, st) != cudaSuccess) return ZP_ERR_CUDA;
  if (R == 0) return ZP_OK;

  CUtensorMap tmK;
  // the K/V pool as {d, 2*Hkv*b rows per (layer, block), layers*num_blocks}; box = one block's
  // b rows of one head, 64 columns
  if (!encode_tmap_3d_bf16(&tmK, pool->base, d, static_cast<uint64_t>(2) * Hkv * b,
                           static_cast<uint64_t>(layers) * pool->num_blocks, static_cast<uint64_t>(d) * 2,
                           static_cast<uint64_t>(2) * Hkv * b * d * 2, 64, b, 1))
    return ZP_ERR_CUDA;
  ApArgs a{};
  a.pool = static_cast<const uint8_t*>(pool->base);
  a.num_blocks = pool->num_blocks;
  a.block_tables = block_tables;
  a.seq_len = meta->seq_len;
  a.out = redund;
  a.err = static_cast<int32_t*>(workspace);
  a.sq = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + 256);
  a.layers = layers;
  a.Hkv = Hkv;
  a.d = d;
  a.b = b;
  a.b_shift = (b == 16) ? 4 : 5;
  a.max_blocks = meta->max_blocks;
  a.L = L;
  a.nt = nt;

  const size_t smem = sizeof(ApSmem) + 1024;
  static std::once_flag once;
  static cudaError_t attr_err = cudaSuccess;
  std::call_once(once, [&] {
    attr_err = cudaFuncSetAttribute(all_pairs_redundancy_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    static_cast<int>(smem));
  });
  if (attr_err != cudaSuccess) return ZP_ERR_CUDA;
  key_sq_norm_kernel<<<static_cast<unsigned>(ctas), kThreadsA, 0, st>>>(a);
  all_pairs_redundancy_kernel<<<static_cast<unsigned>(ctas), kThreadsA, smem, st>>>(tmK, a);
  return cudaGetLastError() == cudaSuccess ? ZP_OK : ZP_ERR_CUDA;
}
