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
// GB300 mapping.  One CTA per (unit, pair of 128-row tiles of t), one CTA per SM, warp-
// specialised: a producer warp TMA-loads the CTA's 256 key rows once (A, 128-byte swizzle, one
// 3-D box per (block, 64-column half)) and streams the unit's 128-key tiles (B) through a
// four-stage ring; an MMA warp issues the two 128 x 128 Gram tiles A_h B^T of each key tile on
// tcgen05 into one of two TMEM buffers; eight epilogue warps (thread = row t) add Gram[t][j] / |k_j|
// over the tile's columns while the next tile is multiplied.  Stages and buffers are handed over
// with mbarriers (full / empty, TMEM full / empty), so copies, MMAs and reductions overlap.  The
// similarity matrix is never stored.  R_all[t] = (acc / |k_t| - cos(k_t, k_t)) / (L-1).  Every
// wait is bounded; a role that gives up raises a flag that ends the others' waits too.
#include <algorithm>
#include <mutex>

#include "zp_internal.h"
#include "zp_ptx.cuh"

namespace zp {
namespace {

constexpr int kTile = 128;        // rows per tile = TMEM lanes = MMA M and N
constexpr int kThreadsA = 128;    // pre-pass: thread = key
constexpr int kEpiWarps = 8;      // epilogue warps: thread = row of the CTA's two row tiles
constexpr int kProdWarp = 8, kMmaWarp = 9;
constexpr int kThreadsW = 320;    // 8 epilogue warps + producer warp + MMA warp
constexpr int kStages = 4;        // B ring depth
constexpr uint32_t kColsA = 512;  // [row half h][buffer u] 128-column fp32 accumulators
constexpr int kMaxTabA = 256;     // block-table entries per request (L <= 4096 at b = 16)
constexpr int kMaxLA = kMaxTabA * 16;
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
  uint8_t A[2][2][kTile * 128];         // [row half][d-half][row][128 B], 128-byte swizzle: the CTA's rows
  uint8_t B[kStages][2][kTile * 128];   // [stage][d-half][row][128 B]: the streamed key tiles
  float inv[kMaxLA];                    // reciprocal key norms of the unit
  int tab[kMaxTabA];
  uint64_t bar_a, full[kStages], empty[kStages], tfull[2], tempty[2];
  uint32_t tmem_base;
  int abort;                            // a role gave up a wait: the others stop waiting
};

__device__ __forceinline__ void ap_record_error(int32_t* err, int code) {
  if (err) atomicCAS(err, 0, code);
}

// Issues the TMA of the 128 key rows [row0, row0 + 128) of the unit into `dst`, only for blocks
// that hold tokens of the sequence, and registers their bytes on `bar` (rows past the
// sequence keep whatever the buffer held; their columns and rows are never used).  Called by a
// whole warp: lane 0 registers the bytes, then lane bi issues the boxes of block bi (one TMA
// instruction stream per lane instead of one thread issuing every box).
__device__ __forceinline__ void load_rows(uint8_t (&dst)[2][kTile * 128], const CUtensorMap* tm, uint64_t* bar,
                                          const ApArgs& a, const int* tab, int layer, int h, int row0, int L,
                                          int lane) {
  const int nhalf = a.d / 64;
  const int blk0 = row0 >> a.b_shift;
  const int nblk = max(0, min(kTile >> a.b_shift, ((L + a.b - 1) >> a.b_shift) - blk0));
  if (lane == 0) mbar_arrive_expect_tx(bar, static_cast<uint32_t>(nblk * a.b * a.d * 2));
  __syncwarp();
  if (lane < nblk)  // nblk <= 128 / 16 = 8
    for (int hd = 0; hd < nhalf; ++hd)
      tma_load_3d(&dst[hd][lane * a.b * 128], tm, bar, hd * 64, h * a.b, layer * a.num_blocks + tab[blk0 + lane]);
  __syncwarp();
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

// Waits for phase `parity` of `bar`; gives up (false) after the time limit, or at once when
// another role has given up.  A thread that gives up raises the flag.
__device__ __forceinline__ bool ap_wait(uint64_t* bar, uint32_t parity, volatile int* abort) {
  const uint32_t addr = smem_u32(bar);
  if (mbar_try_wait(addr, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  while (true) {
    if (mbar_try_wait(addr, parity)) return true;
    if (*abort) return false;
    if (globaltimer_ns() - t0 > kWaitNsA) {
      *abort = 1;
      return false;
    }
  }
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

__global__ void __launch_bounds__(kThreadsW, 1)
    all_pairs_redundancy_kernel(const __grid_constant__ CUtensorMap tmK, const ApArgs a) {
  extern __shared__ uint8_t smem_raw[];
  ApSmem& s = *reinterpret_cast<ApSmem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int np = (a.nt + 1) / 2;  // row-tile pairs per unit
  const int unit = static_cast<int>(blockIdx.x) / np, ip = static_cast<int>(blockIdx.x) % np;
  const int h = unit % a.Hkv, layer = (unit / a.Hkv) % a.layers, r = unit / a.Hkv / a.layers;
  const int row0 = ip * 2 * kTile;  // first row of the pair
  float* const out = a.out + static_cast<int64_t>(unit) * a.L;
  const int L = a.seq_len[r];
  if (L < 0 || L > a.L) {
    if (tid == 0 && ip == 0) ap_record_error(a.err, ZP_ERR_BAD_TABLE);
    return;
  }
  // rows of this pair past the sequence (or all of them) are 0
  for (int t = row0 + tid; t < min(row0 + 2 * kTile, a.L); t += kThreadsW)
    if (t >= L || L < 2) out[t] = 0.0f;
  if (row0 >= L || L < 2) return;

  const int nblk = (L + a.b - 1) >> a.b_shift;
  bool bad = false;
  for (int i = tid; i < nblk; i += kThreadsW) {
    const int e = a.block_tables[static_cast<int64_t>(r) * a.max_blocks + i];
    s.tab[i] = e;
    bad |= (e < 0 || e >= a.num_blocks);
  }
  const int ntc = (L + kTile - 1) / kTile;  // key tiles of the unit
  const float* const sq_unit = a.sq + static_cast<int64_t>(unit) * a.L;
  const bool half1 = row0 + kTile < L;  // the second row tile holds rows of the sequence
  if (tid == 0) {
    mbar_init(&s.bar_a, half1 ? 2 : 1);  // one arrival (with its bytes) per loaded row tile
    for (int st = 0; st < kStages; ++st) {
      mbar_init(&s.full[st], 1);
      mbar_init(&s.empty[st], 1);
    }
    for (int u = 0; u < 2; ++u) {
      mbar_init(&s.tfull[u], 1);
      mbar_init(&s.tempty[u], kEpiWarps);
    }
    s.abort = 0;
    fence_mbar_init();
    prefetch_tensormap(&tmK);
  }
  if (__syncthreads_or(bad)) {
    if (tid == 0) ap_record_error(a.err, ZP_ERR_BAD_TABLE);
    return;
  }
  if (warp == 0) tmem_alloc(&s.tmem_base, kColsA);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = s.tmem_base;
  volatile int* const abort = &s.abort;

  if (warp == kProdWarp) {
    // A: the pair's rows; then the key tiles through the ring (the whole warp: lane 0 waits and
    // registers bytes, every lane issues the boxes of one block)
    load_rows(s.A[0], &tmK, &s.bar_a, a, s.tab, layer, h, row0, L, lane);
    if (half1) load_rows(s.A[1], &tmK, &s.bar_a, a, s.tab, layer, h, row0 + kTile, L, lane);
    int last = -1;  // the last key tile issued
    for (int jt = 0; jt < ntc; ++jt) {
      const int st = jt % kStages;
      bool go = true;
      if (lane == 0 && jt >= kStages) go = ap_wait(&s.empty[st], ((jt / kStages) - 1) & 1, abort);
      if (!__shfl_sync(0xffffffffu, go, 0)) break;
      load_rows(s.B[st], &tmK, &s.full[st], a, s.tab, layer, h, jt * kTile, L, lane);
      last = jt;
    }
    // copies still in flight after a give-up land before the shared memory is released
    if (lane == 0) {
      if (*abort)
        for (int jt = max(0, last - kStages + 1); jt <= last; ++jt)
          mbar_wait_bounded(&s.full[jt % kStages], (jt / kStages) & 1, kWaitNsA);
      mbar_wait_bounded(&s.bar_a, 0, kWaitNsA);
    }
  } else if (warp == kMmaWarp) {
    if (lane == 0) {
      const uint32_t idesc = idesc_bf16_f32(kTile, kTile);
      int issued = 0;
      if (ap_wait(&s.bar_a, 0, abort)) {
        for (int jt = 0; jt < ntc; ++jt) {
          const int st = jt % kStages, u = jt & 1;
          if (!ap_wait(&s.full[st], (jt / kStages) & 1, abort)) break;
          if (jt >= 2 && !ap_wait(&s.tempty[u], ((jt >> 1) - 1) & 1, abort)) break;
          tc_fence_after();
          for (int hh = 0; hh < (half1 ? 2 : 1); ++hh)
            for (int kk = 0; kk < a.d / 16; ++kk) {
              const uint64_t ad = smem_desc_sw128(smem_u32(&s.A[hh][kk >> 2][(kk & 3) * 32]));
              const uint64_t bd = smem_desc_sw128(smem_u32(&s.B[st][kk >> 2][(kk & 3) * 32]));
              mma_bf16(tbase + hh * 2 * kTile + u * kTile, ad, bd, idesc, kk > 0);
            }
          mma_commit(&s.empty[st]);  // the stage is free once these MMAs have read it
          mma_commit(&s.tfull[u]);
          issued = jt + 1;
        }
      }
      // MMAs still in flight after a give-up complete before TMEM is released
      if (*abort && issued > 0) mbar_wait_bounded(&s.tfull[(issued - 1) & 1], ((issued - 1) >> 1) & 1, kWaitNsA);
    }
  } else {
    // epilogue: the reciprocal norms of the unit's keys first (while the first copies and MMAs
    // run), then warp w reads TMEM lanes 32 (w % 4) .. + 31 of row half w / 4
    constexpr int kEpi = kEpiWarps * 32;
    for (int i0 = 0; i0 < ntc * kTile; i0 += 4 * kEpi) {
      float sqv[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int i = i0 + e * kEpi + tid;
        sqv[e] = (i < L) ? sq_unit[i] : 0.0f;
      }
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int i = i0 + e * kEpi + tid;
        if (i < ntc * kTile) s.inv[i] = i < L ? 1.0f / fmaxf(sqrtf(sqv[e]), 1e-12f) : 0.0f;
      }
    }
    asm volatile("bar.sync 1, %0;" ::"n"(kEpi) : "memory");  // the epilogue warps only
    const int hh = warp >> 2, q = warp & 3;
    const int t = row0 + hh * kTile + q * 32 + lane;
    const uint32_t lane_base = static_cast<uint32_t>(q * 32) << 16;
    float acc[4] = {0.0f, 0.0f, 0.0f, 0.0f};
    for (int jt = 0; jt < ntc; ++jt) {
      const int u = jt & 1;
      if (!ap_wait(&s.tfull[u], (jt >> 1) & 1, abort)) break;
      tc_fence_after();
      const int nvalid = min(kTile, L - jt * kTile);  // columns of keys of the sequence
      const float* const ib = &s.inv[jt * kTile];
      uint32_t v4[4][32];
#pragma unroll
      for (int c4 = 0; c4 < 4; ++c4) tmem_ld32_issue(tbase + lane_base + hh * 2 * kTile + u * kTile + c4 * 32, v4[c4]);
      tmem_wait_ld(v4[0]);
      tmem_ld_dep(v4[1]);
      tmem_ld_dep(v4[2]);
      tmem_ld_dep(v4[3]);
      // the accumulator buffer is free as soon as it has been read
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&s.tempty[u]);
#pragma unroll
      for (int c4 = 0; c4 < 4; ++c4) {
        const uint32_t (&v)[32] = v4[c4];
        const float4* ib4 = reinterpret_cast<const float4*>(ib + c4 * 32);
        if (c4 * 32 + 32 <= nvalid) {
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            const float4 w = ib4[e];
            acc[0] = fmaf(__uint_as_float(v[4 * e + 0]), w.x, acc[0]);
            acc[1] = fmaf(__uint_as_float(v[4 * e + 1]), w.y, acc[1]);
            acc[2] = fmaf(__uint_as_float(v[4 * e + 2]), w.z, acc[2]);
            acc[3] = fmaf(__uint_as_float(v[4 * e + 3]), w.w, acc[3]);
          }
        } else {
          // the columns past the sequence may hold anything (the tail of the last block, or
          // an earlier tile): they are skipped, not multiplied by zero
#pragma unroll
          for (int j = 0; j < 32; ++j)
            if (c4 * 32 + j < nvalid) acc[j & 3] = fmaf(__uint_as_float(v[j]), ib[c4 * 32 + j], acc[j & 3]);
        }
      }
    }
    if (!*abort && t < L) {
      const float sq = sq_unit[t];
      const float inv_a = s.inv[t];
      const float sum = (acc[0] + acc[1]) + (acc[2] + acc[3]);
      out[t] = (sum * inv_a - sq * inv_a * inv_a) / static_cast<float>(L - 1);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (tid == 0 && s.abort) ap_record_error(a.err, ZP_ERR_TIMEOUT);
  if (warp == 0) tmem_dealloc(tbase, kColsA);
}

// one CTA per SM: 227 KB of shared memory per CTA at most, 1 KB alignment slack
static_assert(sizeof(ApSmem) + 1024 <= 227 * 1024, "shared memory of one CTA");

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
  const int64_t ctas = static_cast<int64_t>(R) * layers * Hkv * nt;          // pre-pass
  const int64_t pairs = static_cast<int64_t>(R) * layers * Hkv * ((nt + 1) / 2);  // main kernel
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
  static PerDeviceInit attrs;
  const cudaError_t attr_err = attrs.run([&] {
    return cudaFuncSetAttribute(all_pairs_redundancy_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                static_cast<int>(smem));
  });
  if (attr_err != cudaSuccess) return ZP_ERR_CUDA;
  key_sq_norm_kernel<<<static_cast<unsigned>(ctas), kThreadsA, 0, st>>>(a);
  all_pairs_redundancy_kernel<<<static_cast<unsigned>(pairs), kThreadsW, smem, st>>>(tmK, a);
  return cudaGetLastError() == cudaSuccess ? ZP_OK : ZP_ERR_CUDA;
}
