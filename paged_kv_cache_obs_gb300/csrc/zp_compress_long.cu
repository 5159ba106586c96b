// zp_compress_long.cu — the compression pass in several launches, for sequences longer than
// one thread-block cluster covers (4096 < L <= 16384 tokens: the first compression after a very
// long prompt, zh §2.1).  Same operation, readings and results as the fused pass
// (zp_compress.cu), with the cluster's exchanges replaced by kernel boundaries and global
// scratch (the workspace past its first 256 bytes):
//   1. stats:   per 256-key chunk: TMA of K (and once per CTA Q), tcgen05 D1 = Q K^T into
//               TMEM, each window row's (max, exp-sum) over the chunk's visible keys, and the
//               Lightning redundancy of the chunk's keys (warp-level MMA);
//   2. score:   per chunk: every row's normaliser from all chunks' partials, K again, D2 =
//               K Q^T, the attention mass of each key and S = attn + a*G - b*R;
//               (a CTA of these two kernels takes up to 16 consecutive chunks of one unit and
//               copies each chunk's K while the previous chunk's TMEM pass runs)
//   3. select:  per unit: the E = L - k lowest eviction keys by an 8-pass radix select of the
//               64-bit keys (order(S), ~t), destinations by a block-wide scan, and the global
//               scores updated in place (every read before any write);
//   4. compact: per unit: the moved K and V rows, 32 destination slots at a time in
//               increasing order (dst <= src, so a chunk's rows are read before anything lands
//               on them), the next chunk's loads in flight while a chunk is written.
// Every wait is bounded.  A unit with bad metadata or block ids is reported and left untouched.
#include <algorithm>
#include <mutex>

#include "zp_compress_common.cuh"

namespace zp {
namespace {

__device__ __forceinline__ void prefetch_l2(const void* p) {
  asm volatile("prefetch.global.L2 [%0];" ::"l"(reinterpret_cast<uint64_t>(p)));
}

constexpr int kMaxLongL = 16384;
constexpr int kSelThreads = 1024;

struct LongScratch {
  float2* part;  // [units][nch][kRows] (max, exp-sum) of each window row over each chunk
  float* attn;   // [units][L]
  float* red;    // [units][L]
  float* score;  // [units][L]
  int32_t* src;  // [units][L]: source position of each destination slot j < k (-1: a reported unit)
  int nch;       // 256-key chunks per unit at the launch length
  int ngrp;      // CTAs of the stats and score kernels per unit (groups of kChunksPerCta chunks)
};

struct __align__(1024) LongSmem {
  uint8_t K[2][kKeysPerCta * 128];  // [d-half][row][128 B], 128-byte swizzle
  uint8_t Q[2][kRows * 128];
  float2 part[2][kRows];
  float row_off[kRows];
  float inv_n[kKeysPerCta];
  uint64_t bar_tma, bar_mma;
  uint64_t bar_never;  // completed by nothing: the test hook's stalled wait
  uint32_t tmem_base;
};

struct UnitMeta {
  int r, layer, h, L, n_max_r, k_r, slot;
  bool bad;
};

__device__ __forceinline__ UnitMeta unit_meta(const CompressArgs& a, int unit) {
  UnitMeta m;
  m.h = unit % a.Hkv;
  m.r = unit / a.Hkv / a.nl;
  m.layer = a.layer0 + (unit / a.Hkv) % a.nl;
  m.L = a.seq_len[m.r];
  m.n_max_r = a.n_max_req ? a.n_max_req[m.r] : a.n_max;
  m.k_r = (m.n_max_r - 1) * a.b;
  m.slot = a.qslot[m.r];
  m.bad = (m.n_max_r < 2) || (m.n_max_r > a.n_max) || (m.k_r < a.w) || (m.L <= m.k_r) || (m.L > a.L) ||
          m.slot < 0 || m.slot >= a.num_qslots;
  return m;
}

// A CTA of the stats and score kernels takes a group of up to kChunksPerCta consecutive chunks
// of one unit: the window queries, the mbarriers, TMEM and the block ids load once, and each
// chunk's K is copied while the previous chunk's TMEM pass runs.
constexpr int kChunksPerCta = 16;
constexpr int kGroupBlocks = kChunksPerCta * kKeysPerCta / 16;  // block ids of a group (b >= 16)

// TMA of one chunk's K blocks by the 32 lanes of one warp (called by all of them): lane 0
// registers the bytes (and, for the first chunk of a CTA, brings the window queries), then lane
// i issues the boxes of blocks i, i + 32, ...  One thread issuing all of a chunk's 32 boxes in
// sequence stalled its warp for about 6.8k cycles; lanes issuing at once take a fraction of that.
__device__ __forceinline__ void issue_chunk_tma(LongSmem& s, const CUtensorMap* tmK, const CUtensorMap* tmQ,
                                                const CompressArgs& a, const UnitMeta& m, const int* phys, int nblk,
                                                bool with_q, int lane) {
  const int nhalf = a.d / 64;
  if (lane == 0) {
    mbar_arrive_expect_tx(&s.bar_tma, static_cast<uint32_t>(((nblk << a.b_shift) + (with_q ? a.Rw : 0)) * a.d * 2));
    if (with_q)
      for (int hd = 0; hd < nhalf; ++hd)
        tma_load_3d(&s.Q[hd][0], tmQ, &s.bar_tma, hd * 64, m.h * a.Gq, (m.slot * a.layers + m.layer) * a.w);
  }
  __syncwarp();
  for (int bi = lane; bi < nblk; bi += 32)
    for (int hd = 0; hd < nhalf; ++hd)
      tma_load_3d(&s.K[hd][bi * a.b * 128], tmK, &s.bar_tma, hd * 64, m.h * a.b,
                  m.layer * static_cast<int>(a.num_blocks) + phys[bi]);
  __syncwarp();
}

// The K boxes of a chunk whose rows fall in warp `warp`'s 32 rows of the tile (blocks
// [32 warp / b, 32 (warp + 1) / b) of the chunk's nblk), one box per lane, on the already armed
// bar_tma.  Called by all 32 lanes of the warp.
__device__ __forceinline__ void issue_warp_boxes(LongSmem& s, const CUtensorMap* tmK, const CompressArgs& a,
                                                 const UnitMeta& m, const int* phys, int nblk, int warp, int lane) {
  const int nhalf = a.d / 64;
  const int b0 = (warp * 32) >> a.b_shift, b1 = min(nblk, ((warp + 1) * 32) >> a.b_shift);
  if (lane < (b1 - b0) * nhalf) {
    const int bi = b0 + lane / nhalf, hd = lane % nhalf;
    tma_load_3d(&s.K[hd][bi * a.b * 128], tmK, &s.bar_tma, hd * 64, m.h * a.b,
                m.layer * static_cast<int>(a.num_blocks) + phys[bi]);
  }
  __syncwarp();
}

// Chunks [c0, c1) of the unit that this CTA takes (c1 <= c0: none).
__device__ __forceinline__ void group_range(const LongScratch& sc, const UnitMeta& m, int g, int& c0, int& c1) {
  c0 = g * kChunksPerCta;
  c1 = m.bad ? c0 : min(c0 + kChunksPerCta, (m.L + kKeysPerCta - 1) / kKeysPerCta);
}

__device__ __forceinline__ int chunk_keys(const UnitMeta& m, int c) { return min(kKeysPerCta, m.L - c * kKeysPerCta); }

// Common prologue of the stats and score kernels for chunks [c0, c1) (c1 > c0): the group's
// block ids (checked), mbarriers, zeroed Q padding rows.  Returns false if a block id is bad
// (the select kernel reports the unit).
__device__ __forceinline__ bool group_prologue(LongSmem& s, const CompressArgs& a, const UnitMeta& m, int c0, int c1,
                                               int* phys, int tid) {
  const int b0 = (c0 * kKeysPerCta) >> a.b_shift;
  const int nb = (min(m.L, c1 * kKeysPerCta) - c0 * kKeysPerCta + a.b - 1) >> a.b_shift;  // <= kGroupBlocks
  __shared__ int bad_blk;
  if (tid == 0) bad_blk = 0;
  __syncthreads();
  for (int i = tid; i < nb; i += kThreads) {
    const int p = a.block_tables[static_cast<int64_t>(m.r) * a.max_blocks + b0 + i];
    phys[i] = p;
    if (p < 0 || p >= a.num_blocks) bad_blk = 1;
  }
  if (tid == 0) {
    mbar_init(&s.bar_tma, 1);
    mbar_init(&s.bar_mma, 1);
    mbar_init(&s.bar_never, 1);
    fence_mbar_init();
  }
  for (int i = a.Rw * 8 + tid; i < kRows * 8; i += kThreads) {  // padding rows of Q are zero
    reinterpret_cast<uint4*>(s.Q[0])[i] = make_uint4(0, 0, 0, 0);
    reinterpret_cast<uint4*>(s.Q[1])[i] = make_uint4(0, 0, 0, 0);
  }
  fence_proxy_async_smem();
  __syncthreads();
  return !bad_blk;
}

// 1. Row statistics over each chunk and Lightning redundancy of its keys.  Per chunk: D1 on the
//    tensor cores while the warps compute the redundancy (the last reads of K), the next
//    chunk's TMA, then pass 1 over TMEM.
__global__ void __launch_bounds__(kThreads, 2)
    long_stats_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmQ,
                      const CompressArgs a, const LongScratch sc) {
  extern __shared__ uint8_t smem_raw[];
  LongSmem& s = *reinterpret_cast<LongSmem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __shared__ int phys[kGroupBlocks];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int q4 = warp & 3, hh = warp >> 2;
  const int unit = static_cast<int>(blockIdx.x) / sc.ngrp, g = static_cast<int>(blockIdx.x) % sc.ngrp;
  const UnitMeta m = unit_meta(a, unit);
  float2* const pu = sc.part + static_cast<int64_t>(unit) * sc.nch * kRows;
  int c0, c1;
  group_range(sc, m, g, c0, c1);
  // chunks of this group (at the launch length) past the unit's end hold no keys
  if (tid < kRows)
    for (int c = max(c0, c1); c < min(g * kChunksPerCta + kChunksPerCta, sc.nch); ++c)
      pu[c * kRows + tid] = make_float2(-INFINITY, 0.0f);
  if (c1 <= c0) return;
  if (!group_prologue(s, a, m, c0, c1, phys, tid)) {
    if (tid < kRows)
      for (int c = c0; c < c1; ++c) pu[c * kRows + tid] = make_float2(-INFINITY, 0.0f);
    return;
  }
  if (warp == 0) tmem_alloc(&s.tmem_base, kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = s.tmem_base;
  bool ok = true, tma_pending = false;  // (tid 0)
  uint32_t ph_tma = 0, ph_mma = 0;
  if (warp == 0) {
    issue_chunk_tma(s, &tmK, &tmQ, a, m, phys, (chunk_keys(m, c0) + a.b - 1) >> a.b_shift, true, lane);
    tma_pending = true;  // (meaningful in tid 0)
  }
  bool fail = false;
  int boff = 0;  // the chunk's first entry in phys
  for (int c = c0; c < c1 && !fail; ++c) {
    const int t0 = c * kKeysPerCta;
    const int nk = chunk_keys(m, c);
    const int nblk = (nk + a.b - 1) >> a.b_shift;
    const int nblk_next = c + 1 < c1 ? (chunk_keys(m, c + 1) + a.b - 1) >> a.b_shift : 0;
    if (tid == 0) {
      // (the test hook first waits, for a.stall_ns, on a barrier that nothing completes: the
      // wait gives up and the CTA takes its timeout path with the chunk's copy in flight)
      ok = (a.stall_ns == 0 || c != c0 || mbar_wait_bounded(&s.bar_never, 0u, a.stall_ns)) &&
           mbar_wait_bounded(&s.bar_tma, ph_tma, kWaitNs);
      if (ok) {
        ph_tma ^= 1;
        tma_pending = false;
        if (nblk_next > 0) {  // the next chunk's copy; its boxes come from the warps below
          mbar_arrive_expect_tx(&s.bar_tma, static_cast<uint32_t>((nblk_next << a.b_shift) * a.d * 2));
          tma_pending = true;
        }
        tc_fence_after();
        const uint32_t idesc = idesc_bf16_f32(128, (nk + 15) & ~15);
        for (int kk = 0; kk < a.d / 16; ++kk)
          mma_bf16(tbase, smem_desc_sw128(smem_u32(&s.Q[kk >> 2][(kk & 3) * 32])),
                   smem_desc_sw128(smem_u32(&s.K[kk >> 2][(kk & 3) * 32])), idesc, kk > 0);
        mma_commit(&s.bar_mma);
      }
    }
    fail = __syncthreads_or(!ok);  // the chunk's K has landed; D1 runs during the redundancy
    if (fail) break;
    if (warp * 32 < nk) {
      const float red = (a.b == 16) ? warp_lightning_redundancy<16>(s.K, s.inv_n, warp * 32, lane, a.d, t0, m.L)
                                    : warp_lightning_redundancy<32>(s.K, s.inv_n, warp * 32, lane, a.d, t0, m.L);
      if (tid < nk) {
        const int64_t o = static_cast<int64_t>(unit) * a.L + t0 + tid;
        sc.red[o] = red;
        if (a.dbg_redund) a.dbg_redund[((static_cast<int64_t>(m.r) * a.layers + m.layer) * a.Hkv + m.h) * a.L + t0 + tid] = red;
      }
    }
    // This warp's K rows are read (the redundancy); once D1, which reads every row, has
    // completed, they take the next chunk's blocks.  No CTA barrier: each warp issues its own
    // boxes and goes on to pass 1.
    const bool wok = mbar_wait_bounded(&s.bar_mma, ph_mma, kWaitNs);
    ph_mma ^= 1;
    tc_fence_after();
    if (__all_sync(0xffffffffu, wok) && nblk_next > 0) {
      fence_proxy_async_smem();  // this warp's generic reads of K before the copies that replace it
      __syncwarp();
      issue_warp_boxes(s, &tmK, a, m, phys + boff + nblk, nblk_next, warp, lane);
    }
    ok = ok && wok;
    boff += nblk;
    {
      // pass 1: thread = window row i, warp half hh = 128 key columns; keys t <= L-w+i/G_q
      // are visible (columns [0, vlim) of this half to this row, [0, vall) to every row)
      const int i = q4 * 32 + lane;
      const int cbase = hh * 128, ncol = nk - cbase;
      const int vlim = max(0, min(ncol, (a.causal ? (m.L - a.w + i / a.Gq) : (m.L - 1)) - t0 - cbase + 1));
      const int vall = max(0, min(ncol, (a.causal ? (m.L - a.w) : (m.L - 1)) - t0 - cbase + 1));
      const uint32_t tl = tbase + (static_cast<uint32_t>(q4 * 32) << 16) + cbase;
      s.part[hh][i] = row_stats_half(tl, ncol, vlim, vall, a.sl2);
    }
    // every TMEM read of D1 precedes the next chunk's MMA
    tc_fence_before();
    fail = __syncthreads_or(!ok);
    if (fail) break;
    if (tid < kRows) {
      const float2 p0 = s.part[0][tid], p1 = s.part[1][tid];
      float mm = fmaxf(p0.x, p1.x), l = 0.0f;
      if (tid >= a.Rw) mm = -INFINITY;  // a padding row of the MMA, not a window row
      if (mm != -INFINITY) {
        if (p0.y > 0.0f) l += p0.y * ex2((p0.x - mm) * a.sl2);
        if (p1.y > 0.0f) l += p1.y * ex2((p1.x - mm) * a.sl2);
      }
      pu[c * kRows + tid] = make_float2(mm, l);
    }
  }
  if (fail) {
    if (tid < kRows)
      for (int c = c0; c < c1; ++c) pu[c * kRows + tid] = make_float2(-INFINITY, 0.0f);
    if (tid == 0) record_error(a.err, ZP_ERR_TIMEOUT);
  }
  // a copy issued and never seen complete: wait (bounded) before the shared memory goes away
  if (tid == 0 && tma_pending) mbar_wait_bounded(&s.bar_tma, ph_tma, kWaitNs);
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tbase, kTmemCols);
}

// 2. Attention mass of each key (every row normalised over all chunks) and its score S.  Per
//    chunk: D2 (the last read of K), the next chunk's TMA, then pass 2 over TMEM.
__global__ void __launch_bounds__(kThreads, 2)
    long_score_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmQ,
                      const CompressArgs a, const LongScratch sc) {
  extern __shared__ uint8_t smem_raw[];
  LongSmem& s = *reinterpret_cast<LongSmem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __shared__ int phys[kGroupBlocks];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int q4 = warp & 3, hh = warp >> 2;
  const int unit = static_cast<int>(blockIdx.x) / sc.ngrp, g = static_cast<int>(blockIdx.x) % sc.ngrp;
  const UnitMeta m = unit_meta(a, unit);
  int c0, c1;
  group_range(sc, m, g, c0, c1);
  if (c1 <= c0) return;
  if (!group_prologue(s, a, m, c0, c1, phys, tid)) return;
  // every row's normaliser: log2 of its exp-sum over all chunks, relative to its max
  if (tid < kRows) {
    const float2* pu = sc.part + static_cast<int64_t>(unit) * sc.nch * kRows;
    const int nc = (m.L + kKeysPerCta - 1) / kKeysPerCta;
    float M = -INFINITY;
    for (int c = 0; c < nc; ++c) M = fmaxf(M, pu[c * kRows + tid].x);
    float Z = 0.0f;
    if (M != -INFINITY)
      for (int c = 0; c < nc; ++c) {
        const float2 p = pu[c * kRows + tid];
        if (p.y > 0.0f) Z += p.y * ex2((p.x - M) * a.sl2);
      }
    s.row_off[tid] = (tid < a.Rw && Z > 0.0f) ? fmaf(M, a.sl2, lg2(Z)) : INFINITY;
  }
  if (warp == 0) tmem_alloc(&s.tmem_base, kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = s.tmem_base;
  bool ok = true, tma_pending = false;  // (tid 0)
  uint32_t ph_tma = 0, ph_mma = 0;
  if (warp == 0) {
    issue_chunk_tma(s, &tmK, &tmQ, a, m, phys, (chunk_keys(m, c0) + a.b - 1) >> a.b_shift, true, lane);
    tma_pending = true;  // (meaningful in tid 0)
  }
  const int64_t gbase = ((static_cast<int64_t>(m.slot) * a.layers + m.layer) * a.Hkv + m.h) * a.L;
  const int64_t dbase = ((static_cast<int64_t>(m.r) * a.layers + m.layer) * a.Hkv + m.h) * a.L;
  bool fail = false;
  int boff = 0;
  for (int c = c0; c < c1 && !fail; ++c) {
    const int t0 = c * kKeysPerCta;
    const int nk = chunk_keys(m, c);
    const int nblk = (nk + a.b - 1) >> a.b_shift;
    const int kt = t0 + tid;
    // the global score and redundancy of this thread's key load while the chunk's copy runs
    const float g_in = tid < nk ? a.gscores[gbase + kt] : 0.0f;
    const float r_in = tid < nk ? sc.red[static_cast<int64_t>(unit) * a.L + kt] : 0.0f;
    const int nblk_next = c + 1 < c1 ? (chunk_keys(m, c + 1) + a.b - 1) >> a.b_shift : 0;
    if (tid == 0) {
      ok = mbar_wait_bounded(&s.bar_tma, ph_tma, kWaitNs);
      if (ok) {
        ph_tma ^= 1;
        tma_pending = false;
        tc_fence_after();
        const uint32_t idesc = idesc_bf16_f32(128, 128);
        for (int kh = 0; kh < 2 && kh * 128 < nk; ++kh)
          for (int kk = 0; kk < a.d / 16; ++kk)
            mma_bf16(tbase + kh * 128, smem_desc_sw128(smem_u32(&s.K[kk >> 2][kh * 128 * 128 + (kk & 3) * 32])),
                     smem_desc_sw128(smem_u32(&s.Q[kk >> 2][(kk & 3) * 32])), idesc, kk > 0);
        mma_commit(&s.bar_mma);
        ok = mbar_wait_bounded(&s.bar_mma, ph_mma, kWaitNs);
        ph_mma ^= 1;
        if (ok && nblk_next > 0) {  // the next chunk's copy; its boxes come from every warp below
          mbar_arrive_expect_tx(&s.bar_tma, static_cast<uint32_t>((nblk_next << a.b_shift) * a.d * 2));
          tma_pending = true;
        }
      }
    }
    fail = __syncthreads_or(!ok);  // D2 has read K (the only reader in this kernel)
    tc_fence_after();
    if (fail) break;
    // each warp issues the next chunk's boxes for its 32 rows; they land while pass 2 runs
    if (nblk_next > 0) issue_warp_boxes(s, &tmK, a, m, phys + boff + nblk, nblk_next, warp, lane);
    boff += nblk;
    const int wcol = hh * 128 + q4 * 32;
    float attn = 0.0f;
    if (wcol < nk) {
      // thread = key (TMEM lane), columns = window rows; row i sees key kt iff kt <= L-w+i/G_q
      // (every row sees every key of the warp when its last key is at most L - w)
      const uint32_t tl = tbase + (static_cast<uint32_t>(q4 * 32) << 16) + hh * 128;
      const bool all_rows = !a.causal || (t0 + wcol + 31 <= m.L - a.w);
      const int imin = a.causal ? max(0, a.Gq * (kt - (m.L - a.w))) : 0;
      attn = key_mass(tl, a.Rw, all_rows, imin, s.row_off, a.sl2) * a.inv_rw;
    }
    if (tid < nk) {
      const int64_t o = static_cast<int64_t>(unit) * a.L + kt;
      float S = (attn + a.alpha * g_in) - a.beta * r_in;
      if (a.protect_window && kt >= m.L - a.w) S = INFINITY;
      sc.attn[o] = attn;
      sc.score[o] = S;
      if (a.dbg_attn) a.dbg_attn[dbase + kt] = attn;
      if (a.dbg_score) a.dbg_score[dbase + kt] = S;
    }
    // every TMEM read of D2 precedes the next chunk's MMA
    tc_fence_before();
    __syncthreads();
  }
  if (fail && tid == 0) record_error(a.err, ZP_ERR_TIMEOUT);
  if (tid == 0 && tma_pending) mbar_wait_bounded(&s.bar_tma, ph_tma, kWaitNs);
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tbase, kTmemCols);
}

// 3. Selection, destinations and the global-score update, one CTA per unit.
__global__ void __launch_bounds__(kSelThreads) long_select_kernel(const CompressArgs a, const LongScratch sc) {
  constexpr int kPer = kMaxLongL / kSelThreads;  // keys per thread: positions tid + e * kSelThreads
  __shared__ unsigned hist[256];
  __shared__ unsigned long long sh_prefix, sh_key;
  __shared__ unsigned sh_rank, sh_count;
  constexpr int kSelWarps = kSelThreads / 32;
  static_assert(2 * kPer <= 32, "one prefetch lane per row of each array");
  __shared__ int grp_base[kPer * kSelWarps];
  __shared__ int row_total[kPer];
  __shared__ int bad_s;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int unit = blockIdx.x;
  const UnitMeta m = unit_meta(a, unit);
  int32_t* src = sc.src + static_cast<int64_t>(unit) * a.L;
  if (tid == 0) bad_s = m.bad ? 1 : 0;
  __syncthreads();
  if (!m.bad) {  // every block id the unit reads or writes
    const int nsrc = (m.L + a.b - 1) >> a.b_shift;
    for (int i = tid; i < nsrc; i += kSelThreads) {
      const int p = a.block_tables[static_cast<int64_t>(m.r) * a.max_blocks + i];
      if (p < 0 || p >= a.num_blocks) bad_s = 1;
    }
    for (int i = tid; i < m.n_max_r - 1; i += kSelThreads) {
      const int p = a.dst_tables[static_cast<int64_t>(m.r) * a.max_blocks + i];
      if (p < 0 || p >= a.num_blocks) bad_s = 1;
    }
  }
  __syncthreads();
  if (bad_s) {  // reported; the unit keeps its pool rows and global scores
    if (tid == 0) record_error(a.err, ZP_ERR_BAD_TABLE);
    for (int t = tid; t < a.L; t += kSelThreads) src[t] = -1;
    return;
  }
  const int L = m.L, E = L - m.k_r;
  const float* S = sc.score + static_cast<int64_t>(unit) * a.L;
  float* G = a.gscores + ((static_cast<int64_t>(m.slot) * a.layers + m.layer) * a.Hkv + m.h) * a.L;
  const float* attn = sc.attn + static_cast<int64_t>(unit) * a.L;
  // the global scores and attention masses are read only after the selection: ask L2 for them
  // now (lane e of each warp: the 128-byte line of row e, lanes 16 - 31 the masses)
  if (lane < 2 * kPer) {
    const int e = lane % kPer;
    const int t = e * kSelThreads + warp * 32;
    if (t < L) prefetch_l2(lane < kPer ? static_cast<const void*>(G + t) : static_cast<const void*>(attn + t));
  }
  // radix select of the E-th smallest key, 8 bits at a time from the top, until the chosen bin
  // holds a single key (with distinct scores, after 2 or 3 of the 8 passes).  The passes read
  // the scores from registers, loaded once with positions tid + e * kSelThreads (coalesced,
  // every thread busy).  (Aggregating each warp's adds per distinct bin with a match was
  // slower, and so was holding the scores in shared memory, which frees the registers that
  // spill at the 64-register limit of 1024 threads.)
  float sv[kPer];
#pragma unroll
  for (int e = 0; e < kPer; ++e) {
    const int t = tid + e * kSelThreads;
    sv[e] = t < L ? S[t] : 0.0f;
  }
  unsigned long long prefix = 0, mask = 0;
  unsigned rank = static_cast<unsigned>(E);
  for (int pass = 0; pass < 8; ++pass) {
    const int shift = 56 - 8 * pass;
    if (tid < 256) hist[tid] = 0;
    __syncthreads();
#pragma unroll
    for (int e = 0; e < kPer; ++e) {
      const int t = tid + e * kSelThreads;
      if (e * kSelThreads >= L) break;  // uniform over the CTA
      const unsigned long long key = evict_key(sv[e], t);
      if (t < L && (key & mask) == prefix) atomicAdd(&hist[(key >> shift) & 0xFF], 1u);
    }
    __syncthreads();
    if (warp == 0) {
      // the bucket holding the rank-th key: inclusive prefix sums of 8 bins per lane
      unsigned c[8], run = 0;
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        run += hist[lane * 8 + q];
        c[q] = run;
      }
      unsigned incl = run;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const unsigned v = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += v;
      }
      const unsigned before = incl - run;  // keys in the lanes below
      if (before < rank && rank <= incl) {
        int q = 0;
        while (before + c[q] < rank) ++q;
        sh_prefix = prefix | (static_cast<unsigned long long>(lane * 8 + q) << shift);
        sh_rank = rank - (before + (q ? c[q - 1] : 0u));
        sh_count = c[q] - (q ? c[q - 1] : 0u);  // keys in the chosen bin
      }
    }
    __syncthreads();
    prefix = sh_prefix;
    rank = sh_rank;
    mask |= 0xFFull << shift;
    if (sh_count == 1) {  // uniform over the CTA
      // one key left in the bin: it is the rank-th (rank is 1), whatever its lower bits
#pragma unroll
      for (int e = 0; e < kPer; ++e) {
        const int t = tid + e * kSelThreads;
        if (e * kSelThreads >= L) break;  // uniform over the CTA
        const unsigned long long key = evict_key(sv[e], t);
        if (t < L && (key & mask) == prefix) sh_key = key;
      }
      __syncthreads();
      prefix = sh_key;
      break;
    }
  }
  const unsigned long long T = prefix;  // exactly E keys are <= T (keys are distinct)
  // Destinations: j = number of kept keys before t.  Position t = tid + e * kSelThreads stays
  // with the thread that holds its score, so every global access below is coalesced.  A warp
  // ballot per e counts the kept keys of its 32 positions; warp e then scans row e of those
  // counts (positions [e * kSelThreads, (e + 1) * kSelThreads) in order) and the row totals
  // are summed along e in the write loop.
  static_assert(kPer <= kSelWarps, "one warp per row of group counts");
  const unsigned lt_mask = (1u << lane) - 1u;
  unsigned kmask = 0;  // bit e: position tid + e * kSelThreads is kept
#pragma unroll
  for (int e = 0; e < kPer; ++e) {
    const int t = tid + e * kSelThreads;
    const bool kept = t < L && evict_key(sv[e], t) > T;
    kmask |= (kept ? 1u : 0u) << e;
    const unsigned ball = __ballot_sync(0xffffffffu, kept);
    if (lane == 0) grp_base[e * kSelWarps + warp] = __popc(ball);
  }
  __syncthreads();
  if (warp < kPer) {
    const int v = grp_base[warp * kSelWarps + lane];
    int incl = v;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int x = __shfl_up_sync(0xffffffffu, incl, off);
      if (lane >= off) incl += x;
    }
    grp_base[warp * kSelWarps + lane] = incl - v;
    if (lane == 31) row_total[warp] = incl;
  }
  __syncthreads();
  // global scores: every read of the unit's row before any write of it
  float gnew[kPer];
#pragma unroll
  for (int e = 0; e < kPer; ++e) {
    const int t = tid + e * kSelThreads;
    gnew[e] = 0.0f;
    if ((kmask >> e) & 1u) gnew[e] = a.decay * G[t] + attn[t];
  }
  __syncthreads();
  int row_base = 0;  // kept keys in the rows before e
#pragma unroll
  for (int e = 0; e < kPer; ++e) {
    const int t = tid + e * kSelThreads;
    if (e * kSelThreads >= L) break;  // uniform over the CTA
    const bool kept = (kmask >> e) & 1u;
    const unsigned ball = __ballot_sync(0xffffffffu, kept);
    if (kept) {
      const int j = row_base + grp_base[e * kSelWarps + warp] + __popc(ball & lt_mask);
      src[j] = t;
      G[j] = gnew[e];
    }
    if (a.dbg_keep && t < L)
      a.dbg_keep[((static_cast<int64_t>(m.r) * a.layers + m.layer) * a.Hkv + m.h) * a.L + t] = kept;
    row_base += row_total[e];
  }
  __syncthreads();
  for (int t = m.k_r + tid; t < L; t += kSelThreads) G[t] = 0.0f;  // slots past the k survivors
}

// 4. In-place compaction of the moved K and V rows, one CTA per unit, 32 destination slots at a
//    time (small chunks keep the registers low enough for four CTAs per SM).  A row only moves
//    to a lower slot (dst <= src), so the sources of the slots past a chunk all lie past that
//    chunk: chunk by chunk in increasing order, with every read of a chunk before any of its
//    writes, is a safe order, and every chunk is full of kept rows.  The loads of chunk c + 1
//    may run ahead of the writes of chunk c (they read past them), so the kernel keeps two
//    chunks in registers: while chunk c is written, chunk c + 1 is in flight.
//    Per-row byte offsets (source and destination, or -1 for a row that stays) take two
//    dependent loads (the slot's source position, then the block ids).  Every thread computes
//    those of one slot, for a group of kThreads slots (8 chunks) at once, into one of two
//    buffers: group g + 1 during the second chunk of group g, after the barrier that follows
//    the last writes of group g - 1 (the buffer's previous user).  The load latency is then
//    paid once per group instead of once per chunk.
__global__ void __launch_bounds__(kThreads, 4) long_compact_kernel(const CompressArgs a, const LongScratch sc) {
  constexpr int kRowsC = 32;                                  // destination slots per chunk
  constexpr int kPerC = kRowsC * 2 * 128 / 8 / kThreads;      // 16-byte pieces per thread at d = 128
  constexpr int kChunksG = kThreads / kRowsC;                 // chunks per group of offsets
  __shared__ long long src_off[2][kThreads], dst_off[2][kThreads];
  const int tid = threadIdx.x;
  const int unit = blockIdx.x;
  const UnitMeta m = unit_meta(a, unit);
  if (m.bad) return;
  const int32_t* src = sc.src + static_cast<int64_t>(unit) * a.L;
  const int32_t* src_tab = a.block_tables + static_cast<int64_t>(m.r) * a.max_blocks;
  const int32_t* dst_tab = a.dst_tables + static_cast<int64_t>(m.r) * a.max_blocks;
  uint8_t* const head_base = a.pool + static_cast<size_t>(m.layer) * static_cast<size_t>(a.num_blocks) * a.block_bytes +
                             static_cast<size_t>(m.h) * a.b * a.row_bytes;
  const int bm = a.b - 1;
  const int half = a.d / 8;        // 16-byte pieces of a K (or V) row
  const int pieces = 2 * half;     // K then V
  const int total = kRowsC * pieces;
  const int nchunks = (m.k_r + kRowsC - 1) / kRowsC;
  auto offsets = [&](int g) {  // every thread: the byte offsets of slot g * kThreads + tid
    const int j = g * kThreads + tid;
    long long so = -1, dso = -1;
    if (j < m.k_r) {
      const int t = src[j];  // -1 for a reported unit
      if (t >= 0) {
        const int sb = src_tab[t >> a.b_shift], db = dst_tab[j >> a.b_shift];
        if (sb != db || (t & bm) != (j & bm)) {
          so = static_cast<long long>(static_cast<uint32_t>(sb)) * a.block_bytes + static_cast<uint32_t>(t & bm) * a.row_bytes;
          dso = static_cast<long long>(static_cast<uint32_t>(db)) * a.block_bytes + static_cast<uint32_t>(j & bm) * a.row_bytes;
        }
      }
    }
    src_off[g & 1][tid] = so;
    dst_off[g & 1][tid] = dso;
  };
  auto refill = [&](int c) {  // during the second chunk of group g >= 1: group g + 1
    if (c % kChunksG == 1 && c > kChunksG) {
      const int g = c / kChunksG + 1;
      if (g * kThreads < m.k_r) offsets(g);
    }
  };
  auto load = [&](uint4 (&v)[kPerC], int c) {
    const long long* so_c = &src_off[(c / kChunksG) & 1][(c % kChunksG) * kRowsC];
#pragma unroll
    for (int q = 0; q < kPerC; ++q) {
      const int i = tid + q * kThreads;
      v[q] = make_uint4(0u, 0u, 0u, 0u);
      if (i < total) {
        const int row = i / pieces, pc = i % pieces;
        const long long so = so_c[row];
        if (so >= 0) v[q] = *reinterpret_cast<const uint4*>(head_base + so + (pc >= half ? a.kv_bytes : 0u) + (pc % half) * 16);
      }
    }
  };
  auto store = [&](const uint4 (&v)[kPerC], int c) {
    const long long* dso_c = &dst_off[(c / kChunksG) & 1][(c % kChunksG) * kRowsC];
#pragma unroll
    for (int q = 0; q < kPerC; ++q) {
      const int i = tid + q * kThreads;
      if (i < total) {
        const int row = i / pieces, pc = i % pieces;
        const long long dso = dso_c[row];
        if (dso >= 0) *reinterpret_cast<uint4*>(head_base + dso + (pc >= half ? a.kv_bytes : 0u) + (pc % half) * 16) = v[q];
      }
    }
  };
  if (nchunks == 0) return;
  offsets(0);
  if (kThreads < m.k_r) offsets(1);
  __syncthreads();
  uint4 va[kPerC], vb[kPerC];
  load(va, 0);
  for (int c = 0; c < nchunks; c += 2) {
    // chunk c is in va
    if (c + 1 < nchunks) load(vb, c + 1);
    refill(c);
    __syncthreads();  // every read of chunk c precedes every write landing on it
    store(va, c);
    if (c + 1 >= nchunks) break;
    // chunk c + 1 is in vb
    if (c + 2 < nchunks) load(va, c + 2);
    refill(c + 1);
    __syncthreads();
    store(vb, c + 1);
  }
}

static_assert(sizeof(LongSmem) + 1024 <= (228 * 1024 - 2 * 1024) / 2, "two CTAs per SM");

}  // namespace

size_t compress_long_scratch_bytes(int64_t units, int L) {
  const int64_t nch = (L + kKeysPerCta - 1) / kKeysPerCta;
  return static_cast<size_t>(units) * (static_cast<size_t>(nch) * kRows * sizeof(float2) + static_cast<size_t>(L) * 16);
}

zp_status launch_compress_long(const CUtensorMap& tmK, const CUtensorMap& tmQ, const CompressArgs& a, void* scratch,
                               cudaStream_t st) {
  if (a.L > kMaxLongL) return ZP_ERR_UNSUPPORTED;
  const int64_t units = static_cast<int64_t>(a.R) * a.nl * a.Hkv;
  LongScratch sc{};
  sc.nch = (a.L + kKeysPerCta - 1) / kKeysPerCta;
  sc.ngrp = (sc.nch + kChunksPerCta - 1) / kChunksPerCta;
  uint8_t* p = static_cast<uint8_t*>(scratch);
  sc.part = reinterpret_cast<float2*>(p);
  p += static_cast<size_t>(units) * sc.nch * kRows * sizeof(float2);
  sc.attn = reinterpret_cast<float*>(p);
  p += static_cast<size_t>(units) * a.L * 4;
  sc.red = reinterpret_cast<float*>(p);
  p += static_cast<size_t>(units) * a.L * 4;
  sc.score = reinterpret_cast<float*>(p);
  p += static_cast<size_t>(units) * a.L * 4;
  sc.src = reinterpret_cast<int32_t*>(p);
  if (units * sc.nch >= (int64_t(1) << 31)) return ZP_ERR_UNSUPPORTED;
  const size_t smem = sizeof(LongSmem) + 1024;
  static PerDeviceInit attrs;
  const cudaError_t attr = attrs.run([&] {
    cudaError_t e =
        cudaFuncSetAttribute(long_stats_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(long_score_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    return e;
  });
  if (attr != cudaSuccess) return ZP_ERR_CUDA;
  const unsigned chunks = static_cast<unsigned>(units * sc.ngrp);
  long_stats_kernel<<<chunks, kThreads, smem, st>>>(tmK, tmQ, a, sc);
  long_score_kernel<<<chunks, kThreads, smem, st>>>(tmK, tmQ, a, sc);
  long_select_kernel<<<static_cast<unsigned>(units), kSelThreads, 0, st>>>(a, sc);
  long_compact_kernel<<<static_cast<unsigned>(units), kThreads, 0, st>>>(a, sc);
  return cudaGetLastError() == cudaSuccess ? ZP_OK : ZP_ERR_CUDA;
}

}  // namespace zp
