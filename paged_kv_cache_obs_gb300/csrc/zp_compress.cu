// zp_compress.cu — fused compression pass of Compressed PagedAttention for sm_103a.
//
// Operation (Zipage summaries on gist.science: zh §2.1 core mechanism and Lightning Redundancy
// Score, zh §2.2 prefix-cache compatibility, zh §2.3 cross-layer parallel compression, fr §2.A
// window always kept).  Per unit u = (request r, layer l, kv head h) with L cached tokens
// (L = n_max*b at the decode trigger, more after a long prefill) and k = (n_max-1)*b:
//   attn[t] = mean_{rows (i,g)} softmax_t(scale*<q_{i,g}, k_t>)   (row i = position L-w+i)
//   R[t]    = mean_{j in block(t), j != t} cos(k_t, k_j)           (Lightning redundancy)
//   S[t]    = attn[t] + alpha*G[t] - beta*R[t]                     (+inf on the protected window)
//   keep the k best (S desc, t asc), copy survivor j to slot j of the dst table,
//   G'[j] = decay*G[src_j] + attn[src_j], G'[k..L) = 0.
//
// GB300 mapping.  Persistent thread-block clusters of C = ceil(L/256) CTAs (up to 8 at two
// CTAs per SM, up to 16 at one) take units from a global counter; CTA c owns the 256 logical
// slots [256c, 256c+256).  Per unit each CTA:
//   1. TMA-loads its K rows (paged gather: one 3-D box per (block, 64-column half)) and the
//      unit's w*G_q window queries into 128-byte-swizzled shared memory.
//   2. tcgen05 MMA D1 = Q K^T (M=128 query rows, N=256 keys) into TMEM; each thread owns one
//      query row and reduces its row max / exp-sum without shuffles (pass 1).
//   3. Sends the per-row (max, sum) partials to every CTA of the cluster as st.async stores
//      counted on the receiver's mbarrier; meanwhile each warp computes the Lightning
//      redundancy of its 32 keys with warp-level MMA (block Gram, diagonal = squared norms).
//   4. MMA D2 = K Q^T (M=128 keys, N=128 rows): each thread owns one key and sums its
//      normalised probabilities over the window rows without shuffles (pass 2).
//   5. Selection of the E = L-k lowest (S asc, t desc) keys: per-warp bitonic sorts and merge
//      trees (E <= 32), or per-warp sorts merged by rank into a sorted list per CTA and ranks
//      by binary search in local copies of every CTA's sorted list (E > 32); every CTA
//      derives the same eviction set.
//   6. V rows are staged (shared memory and registers) before a cluster barrier that separates
//      every read of the unit from every write (compaction is in place, dst <= src); K rows are
//      written from shared memory, V rows from the staging, G' from registers.
// All waits are bounded; a failed wait or a bad table makes the whole unit skip its writes.
#include <cstdio>
#include <algorithm>
#include <mutex>

#include "zp_compress_common.cuh"

namespace zp {
namespace {



template <int MAXC>
struct __align__(1024) SmemT {
  uint8_t K[2][kKeysPerCta * 128];  // [d-half][row][128 B], 128-byte swizzle
  uint8_t Q[2][kRows * 128];
  // key lists that fit the row-partial area beside this CTA's own sorted list
  static constexpr int kU1Copies = MAXC * kRows / kKeysPerCta - 1;
  union {
    float2 part[2][kRows];          // pass-1 (max, sum) per column half
    unsigned long long lists[(MAXC - 2) * 32];  // cluster-level merge of the eviction candidates
    unsigned long long copy[kKeysPerCta];       // local copy of another CTA's sorted keys
  } u0;
  union {
    float2 recv[MAXC][kRows];                   // (max, sum) partials of every CTA
    struct {
      unsigned long long key[kKeysPerCta];      // eviction keys of this CTA (sorted on the many-eviction path)
      unsigned long long copy[kU1Copies][kKeysPerCta];  // local copies of other CTAs' sorted keys
    } sel;
  } u1;
  unsigned long long cand_recv[MAXC * 32];  // sorted bottom-32 list of every CTA
  int status_recv[MAXC];
  float row_off[kRows];
  int evict_pos[kMaxEvict];
  int src_tab[max_table(MAXC)];
  int dst_tab[max_table(MAXC)];
  int dst_of[kKeysPerCta];          // destination slot of each key that moves, else -1
  float inv_n[kKeysPerCta];         // reciprocal key norms (Gram diagonal)
  uint64_t bar_tma;
  uint64_t bar_mma;
  uint64_t bar_v;
  uint64_t bar_rs;                  // row statistics of every CTA of the cluster have landed
  uint32_t tmem_base;
  int next_unit[2];                 // unit after the current one, pushed by cluster rank 0
  int kept_recv[MAXC];              // kept keys of every CTA (many-eviction path)
  int warp_kept[kThreads / 32];
};

// two CTAs per SM: 228 KB of shared memory per SM, 1 KB of it reserved per CTA, plus the
// 1 KB alignment slack of the dynamic allocation
static_assert(sizeof(SmemT<8>) + 1024 <= (228 * 1024 - 2 * 1024) / 2, "8-CTA clusters: two CTAs per SM");
static_assert(sizeof(SmemT<16>) + 1024 <= 227 * 1024, "16-CTA clusters: one CTA per SM");
static_assert(sizeof(SmemT<8>::cand_recv) % (kKeysPerCta * 8) == 0, "the candidate lists hold whole key lists");

// Local key-list buffers of the many-eviction selection: the row-partial area beside the
// CTA's own list, the candidate lists and u0.  None of them is used by anything else between
// the sort and barrier #2 on that path (the candidate lists and the u0 merge belong to the
// few-eviction path; the row partials of the unit have been combined, and those of the next
// unit only arrive after barrier #2).
template <int MAXC>
constexpr int kSelBufs = SmemT<MAXC>::kU1Copies + MAXC / 8 + 1;

template <int MAXC>
__device__ __forceinline__ unsigned long long* sel_buf(SmemT<MAXC>& s, int i) {
  constexpr int nu1 = SmemT<MAXC>::kU1Copies, nc = MAXC / 8;
  if (i < nu1) return s.u1.sel.copy[i];
  if (i < nu1 + nc) return s.cand_recv + (i - nu1) * kKeysPerCta;
  return s.u0.copy;
}

// Sorts one 64-bit key per lane ascending across the warp (bitonic network).
__device__ __forceinline__ unsigned long long warp_sort32(unsigned long long x, int lane) {
#pragma unroll
  for (int k = 2; k <= 32; k <<= 1) {
#pragma unroll
    for (int j = k >> 1; j > 0; j >>= 1) {
      const unsigned long long y = __shfl_xor_sync(0xffffffffu, x, j);
      const bool take_min = ((lane & j) == 0) == ((lane & k) == 0);
      const unsigned long long lo = x < y ? x : y, hi = x < y ? y : x;
      x = take_min ? lo : hi;
    }
  }
  return x;
}

// The 32 smallest of two ascending 32-key lists (one key per lane each), ascending: the
// elementwise minimum of a and reversed b is bitonic and holds them; a bitonic merge sorts it.
__device__ __forceinline__ unsigned long long warp_merge_low32(unsigned long long a, unsigned long long b,
                                                               int lane) {
  const unsigned long long br = __shfl_sync(0xffffffffu, b, 31 - lane);
  unsigned long long x = a < br ? a : br;
#pragma unroll
  for (int j = 16; j > 0; j >>= 1) {
    const unsigned long long y = __shfl_xor_sync(0xffffffffu, x, j);
    const unsigned long long lo = x < y ? x : y, hi = x < y ? y : x;
    x = ((lane & j) == 0) ? lo : hi;
  }
  return x;
}

template <int MAXC>
__global__ void __launch_bounds__(kThreads, MAXC <= 8 ? 2 : 1)
    compress_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmQ,
                    const CompressArgs a) {
  using Smem = SmemT<MAXC>;
  extern __shared__ uint8_t smem_raw[];
  Smem& s = *reinterpret_cast<Smem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int q4 = warp & 3, hh = warp >> 2;  // TMEM lane quarter, key/column half
  const int C = static_cast<int>(cluster_nctarank());
  const int c = static_cast<int>(cluster_ctarank());
  // La: the longest sequence of the call (row length of the global scores); Lx: the keys this
  // launch's clusters cover (cluster size, TMA/MMA shapes; La unless the requests are grouped
  // by length); L: this unit's own sequence length (all masking and selection)
  const int La = a.L, Lx = a.Lc, b = a.b, d = a.d, w = a.w, Rw = a.Rw, Gq = a.Gq;
  const int bs = a.b_shift, bm = b - 1;  // b is a power of two: t / b = t >> bs, t % b = t & bm
  const int t0 = c * kKeysPerCta;
  const int nk_l = min(kKeysPerCta, Lx - t0);          // keys of this CTA at the launch length
  const int nblk_l = (nk_l + bm) >> bs;                // blocks loaded (a partial last block whole)
  const int n_mma = (nk_l + 15) & ~15;                 // MMA N over those keys
  const int nhalf = d / 64;
  // the launch's requests: all of them, or one length group (positions [rbase, rbase + count)
  // of the grouped order)
  const int rbase = a.bucket ? a.bucket[0] : 0;
  const int num_units = (a.bucket ? a.bucket[1] : a.R) * a.nl * a.Hkv;
  const int cluster_id = static_cast<int>(blockIdx.x) / C;  // the C CTAs of a cluster are consecutive in x
  const int num_clusters = static_cast<int>(gridDim.x) / C;

  // ---------------------------------------------------------------- once per CTA --------
  if (tid == 0) {
    mbar_init(&s.bar_tma, 1);
    mbar_init(&s.bar_mma, 1);
    mbar_init(&s.bar_v, 1);
    mbar_init(&s.bar_rs, 1);
    fence_mbar_init();
    prefetch_tensormap(&tmK);
    prefetch_tensormap(&tmQ);
  }
  __syncwarp();
  if (warp == 0) tmem_alloc(&s.tmem_base, kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = s.tmem_base;
  // mbarrier phases, tracked by the waiting thread (tid 0): every unit completes bar_tma once,
  // bar_v once (unless skipped) and bar_mma three times (unless skipped)
  uint32_t ph_tma = 0, ph_mma = 0, ph_v = 0;
  // bar_rs completes once per unit that is not skipped; every thread tracks its phase (skip is
  // uniform across the cluster)
  uint32_t ph_rs = 0;

  // Persistent clusters: cluster i starts with unit i and then takes the next unused unit from
  // a global counter (fetched by cluster rank 0, broadcast through shared memory); a unit is
  // (request, layer, kv head) with the kv head fastest.
  int iter = 0;
  for (int unit = cluster_id; unit < num_units; ++iter) {
  const int h = unit % a.Hkv;
  const int r = a.req_order ? a.req_order[rbase + unit / a.Hkv / a.nl] : unit / a.Hkv / a.nl;
  const int layer = a.layer0 + (unit / a.Hkv) % a.nl;
  uint8_t* const head_base = a.pool + static_cast<size_t>(layer) * static_cast<size_t>(a.num_blocks) * a.block_bytes +
                             static_cast<size_t>(h) * b * a.row_bytes;

  // ---- set-up of the unit.  Warp 0 issues the TMA of K and Q straight away from the table
  //      entries it reads itself; a block id outside the pool only makes TMA fill zeros, and
  //      the unit is then skipped after validation below (waiting for the copies).
  const int slot = a.qslot[r];
  bool tma_pending = false, v_pending = false;  // (tid 0) copies issued and not yet waited for
  if (warp == 0) {
    // lane 0 registers the bytes, then every lane issues the boxes of its own block(s)
    if (lane == 0) {
      mbar_arrive_expect_tx(&s.bar_tma, static_cast<uint32_t>(((nblk_l << bs) + Rw) * d * 2));
      for (int hd = 0; hd < nhalf; ++hd)
        tma_load_3d(&s.Q[hd][0], &tmQ, &s.bar_tma, hd * 64, h * Gq, (slot * a.layers + layer) * w);
      tma_pending = true;
    }
    __syncwarp();
    const int32_t* trow = a.block_tables + static_cast<int64_t>(r) * a.max_blocks + (t0 >> bs);
    for (int bi = lane; bi < nblk_l; bi += 32) {
      const int phys = trow[bi];
      for (int hd = 0; hd < nhalf; ++hd)
        tma_load_3d(&s.K[hd][bi * b * 128], &tmK, &s.bar_tma, hd * 64, h * b,
                    layer * static_cast<int>(a.num_blocks) + phys);
    }
    __syncwarp();
  }
  // cluster rank 0 fetches the unit after this one now and sends it to every CTA with its
  // status before barrier #2 (the atomic's latency overlaps the unit's work)
  int next_fetch = 0;
  if (c == 0 && tid == 0) next_fetch = num_clusters + atomicAdd(a.work, 1);

  // Validate the request's metadata; every CTA of the cluster sees the same values, so they
  // all take the same decision without communicating.  A request holds L cached tokens with
  // k < L <= Lx (L = n_max*b at the decode trigger; more after a long prefill).
  const int L = a.seq_len[r];
  // the request's block budget (all requests share n_max unless per-request budgets are given)
  const int n_max_r = a.n_max_req ? a.n_max_req[r] : a.n_max;
  // Every table entry the launch may use is loaded now, independently of L and of the budget,
  // so that these loads overlap the two above; only the request's own entries are checked.
  const int nblk_a = (Lx + bm) >> bs;  // <= max_table(MAXC) <= kThreads
  const int sb = tid < nblk_a ? a.block_tables[static_cast<int64_t>(r) * a.max_blocks + tid] : 0;
  const int db = tid < a.n_max - 1 ? a.dst_tables[static_cast<int64_t>(r) * a.max_blocks + tid] : 0;
  const int k_r = (n_max_r - 1) * b;                 // tokens this request keeps per head
  bool bad = (n_max_r < 2) || (n_max_r > a.n_max) || (k_r < w) || (L <= k_r) || (L > Lx) || slot < 0 ||
             slot >= a.num_qslots;
  if (tid < nblk_a) {
    s.src_tab[tid] = sb;
    if (tid < ((L + bm) >> bs)) bad |= (sb < 0 || sb >= a.num_blocks);
  }
  if (tid < a.n_max - 1) {
    s.dst_tab[tid] = db;
    if (tid < n_max_r - 1) bad |= (db < 0 || db >= a.num_blocks);
  }
  const int nk = max(0, min(kKeysPerCta, L - t0));   // this unit's keys in this CTA
  const int E = L - k_r;                              // tokens to evict per head
  // Zero the padding rows of Q (never touched by the TMA box; the V staging of the previous
  // unit may have used them).
  for (int i = Rw * 8 + tid; i < kRows * 8; i += kThreads) {
    const int row = i >> 3, ch = i & 7;
    reinterpret_cast<uint4*>(s.Q[0])[row * 8 + ch] = make_uint4(0, 0, 0, 0);
    reinterpret_cast<uint4*>(s.Q[1])[row * 8 + ch] = make_uint4(0, 0, 0, 0);
  }
  fence_proxy_async_smem();
  tc_fence_before();
  const bool skip = __syncthreads_or(bad);
  tc_fence_after();
  if (skip && tid == 0 && c == 0) record_error(a.err, ZP_ERR_BAD_TABLE);
  // every CTA of the cluster (this one included) delivers 128 row partials of 8 bytes here
  if (!skip && tid == 0) mbar_arrive_expect_tx(&s.bar_rs, static_cast<uint32_t>(C * kRows * 8));

  const int kt = t0 + tid;  // the key this thread owns from pass 2 on
  const bool key_valid = tid < nk;
  float g_in = 0.0f;
  float attn = 0.0f, red = 0.0f, S = 0.0f;
  bool ok = true;  // outcome of the bounded waits, meaningful in the waiting thread (tid 0)

  // ---- step 1: TMA of K and Q, then D1 = Q K^T (M = 128 window rows, N = nk keys).  Only
  //      thread 0 waits on the mbarriers; the others block on the CTA barrier below.
  if (!skip) {
    if (key_valid) g_in = a.gscores[((static_cast<int64_t>(slot) * a.layers + layer) * a.Hkv + h) * La + kt];
    if (tid == 0) {
      ok = mbar_wait_bounded(&s.bar_tma, ph_tma, kWaitNs);
      if (ok) {
        ph_tma ^= 1;
        tma_pending = false;
      }
      tc_fence_after();
      const uint32_t idesc = idesc_bf16_f32(128, n_mma);
      for (int kk = 0; kk < d / 16; ++kk) {
        const uint64_t ad = smem_desc_sw128(smem_u32(&s.Q[kk >> 2][(kk & 3) * 32]));
        const uint64_t bd = smem_desc_sw128(smem_u32(&s.K[kk >> 2][(kk & 3) * 32]));
        mma_bf16(tbase, ad, bd, idesc, kk > 0);
      }
      mma_commit(&s.bar_mma);
      ok = mbar_wait_bounded(&s.bar_mma, ph_mma, kWaitNs) && ok;
      ph_mma ^= 1;
    }
  }
  bool fail = __syncthreads_or(!ok);
  tc_fence_after();

  // ---- step 2 (pass 1): per-row max and exp-sum over this CTA's keys.  Thread = window row
  //      (TMEM lane), warp half hh = 128 key columns; two 32-column loads per wait.  A group of
  //      32 columns that every row sees completely takes the unpredicated path; the others
  //      compare the column with this row's visibility limit (one compare per element).
  if (!skip) {
    const int i = q4 * 32 + lane;
    const int cbase = hh * 128;
    const int ncol = nk - cbase;                         // valid columns of this half (may be <= 0)
    // columns [0, vlim) of this half are visible to this row, [0, vall) to every row
    const int vlim = max(0, min(ncol, (a.causal ? (L - w + i / Gq) : (L - 1)) - t0 - cbase + 1));
    const int vall = max(0, min(ncol, (a.causal ? (L - w) : (L - 1)) - t0 - cbase + 1));
    const uint32_t tl = tbase + (static_cast<uint32_t>(q4 * 32) << 16) + cbase;
    // rows without a visible key get m = -inf and l = 0; padding rows are dropped below
    s.u0.part[hh][i] = row_stats_half(tl, ncol, vlim, vall, a.sl2);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();

  // ---- step 3: D2 = K Q^T per 128-key half into TMEM (D1 fully read) while the row partials
  //      go to every CTA of the cluster as asynchronous stores that count on its bar_rs (no
  //      cluster barrier).  The Lightning redundancy (warp-level MMA on K in shared memory) is
  //      computed while they travel.
  if (!skip) {
    if (tid == 0) {
      const uint32_t idesc = idesc_bf16_f32(128, 128);
      for (int kh = 0; kh < 2 && kh * 128 < nk_l; ++kh)
        for (int kk = 0; kk < d / 16; ++kk) {
          const uint64_t ad = smem_desc_sw128(smem_u32(&s.K[kk >> 2][kh * 128 * 128 + (kk & 3) * 32]));
          const uint64_t bd = smem_desc_sw128(smem_u32(&s.Q[kk >> 2][(kk & 3) * 32]));
          mma_bf16(tbase + kh * 128, ad, bd, idesc, kk > 0);
        }
      mma_commit(&s.bar_mma);
    }
    if (tid < kRows) {
      const float2 p0 = s.u0.part[0][tid], p1 = s.u0.part[1][tid];
      float m = fmaxf(p0.x, p1.x), l = 0.0f;
      if (tid >= Rw) m = -INFINITY;  // padding row of the MMA, not a window row
      if (m != -INFINITY) {
        if (p0.y > 0.0f) l += p0.y * ex2((p0.x - m) * a.sl2);
        if (p1.y > 0.0f) l += p1.y * ex2((p1.x - m) * a.sl2);
      }
      const uint32_t local = smem_u32(&s.u1.recv[c][tid]), lbar = smem_u32(&s.bar_rs);
      for (int dst = 0; dst < C; ++dst) st_async_v2(mapa(local, dst), m, l, mapa(lbar, dst));
    }
  }
  const int wcol = hh * 128 + q4 * 32;  // first key of this warp (TMEM lanes of pass 2)
  if (!skip && warp * 32 < nk) {
    red = (b == 16) ? warp_lightning_redundancy_rolled<16>(s.K, s.inv_n, warp * 32, lane, d, t0, L)
                    : warp_lightning_redundancy_rolled<32>(s.K, s.inv_n, warp * 32, lane, d, t0, L);
  }

  if (!skip) {
    if (tid < kRows) {
      // every CTA's row partials have landed (each combining thread waits for itself)
      ok = mbar_wait_bounded_cluster(&s.bar_rs, ph_rs, kWaitNs) && ok;
      float M = -INFINITY;
      for (int cc = 0; cc < C; ++cc) M = fmaxf(M, s.u1.recv[cc][tid].x);
      float Lsum = 0.0f;
      if (M != -INFINITY)
        for (int cc = 0; cc < C; ++cc) {
          const float2 p = s.u1.recv[cc][tid];
          if (p.y > 0.0f) Lsum += p.y * ex2((p.x - M) * a.sl2);
        }
      s.row_off[tid] = (tid < Rw && Lsum > 0.0f) ? fmaf(M, a.sl2, lg2(Lsum)) : INFINITY;
    }
    ph_rs ^= 1;
    if (tid == 0) {
      ok = mbar_wait_bounded(&s.bar_mma, ph_mma, kWaitNs) && ok;
      ph_mma ^= 1;
    }
  }
  fail |= __syncthreads_or(!ok);
  tc_fence_after();

  // ---- step 5: Q is no longer needed: stage V rows [0, min(128, nk)) into its place by bulk
  //      copies (one per block), then pass 2, then V rows [128, nk) into registers.  All of it
  //      completes before the second cluster barrier, which therefore also separates every
  //      read of the unit from every write.
  uint8_t* const vstage = &s.Q[0][0];
  const int nv0 = min(128, nk);
  if (!skip && tid == 0 && nv0 > 0) {
    const int nvb = (nv0 + bm) >> bs;  // whole blocks (a partial last block is copied whole)
    mbar_arrive_expect_tx(&s.bar_v, static_cast<uint32_t>(nvb << bs) * a.row_bytes);
    for (int bi = 0; bi < nvb; ++bi) {
      const uint8_t* src = head_base + row_off_bytes(a, s.src_tab[(t0 >> bs) + bi], 1, 0);
      bulk_load(vstage + static_cast<size_t>(bi) * b * a.row_bytes, src, static_cast<uint32_t>(b) * a.row_bytes,
                &s.bar_v);
    }
    v_pending = true;
  }
  __syncwarp();  // warp 0 reconverges before the collective TMEM loads
  if (!skip) {
    // pass 2: attention mass of this key over the window rows.  Thread = key (TMEM lane),
    // columns = window rows; rows beyond R_w have row_off = +inf and add 0.
    if (wcol < nk) {
      const uint32_t tl = tbase + (static_cast<uint32_t>(q4 * 32) << 16) + hh * 128;
      const bool all_rows = !a.causal || (t0 + wcol + 31 <= L - w);
      const int imin = a.causal ? max(0, Gq * (kt - (L - w))) : 0;
      attn = key_mass(tl, Rw, all_rows, imin, s.row_off, a.sl2) * a.inv_rw;
    }
    S = (attn + a.alpha * g_in) - a.beta * red;
    if (a.protect_window && kt >= L - w) S = INFINITY;
    if (key_valid) {
      const int64_t o = ((static_cast<int64_t>(r) * a.layers + layer) * a.Hkv + h) * La + kt;
      if (a.dbg_attn) a.dbg_attn[o] = attn;
      if (a.dbg_redund) a.dbg_redund[o] = red;
      if (a.dbg_score) a.dbg_score[o] = S;
    }
  }
  // V rows [128, nk): warp w holds rows 128 + 16w .. 128 + 16w + 15 (rpi rows per load)
  const int cpr = d / 8, rpi = 32 / cpr;
  uint4 vreg[8];
#pragma unroll
  for (int it = 0; it < 8; ++it) {
    vreg[it] = make_uint4(0, 0, 0, 0);
    const int row = 128 + warp * 16 + it * rpi + lane / cpr, ch = lane % cpr;
    if (!skip && it * rpi < 16 && row < nk) {
      const int t = t0 + row;
      vreg[it] = *reinterpret_cast<const uint4*>(head_base + row_off_bytes(a, s.src_tab[t >> bs], 1, t & bm) + ch * 16);
    }
  }

  // ---- step 6: selection.  The E evicted keys are the E smallest eviction keys of the
  //      cluster (E = L - k, the same in every CTA of the cluster).
  unsigned long long* const lst = s.u1.sel.key;
  const unsigned long long mykey =
      (!skip && key_valid) ? evict_key(S, kt) : (~0ull - static_cast<unsigned long long>(tid));
  bool evicted = false;
  if (E <= 32) {
    // Each warp sorts its 32 keys; the 8 sorted lists merge pairwise (bottom 32 of each pair)
    // in a 3-level tree; the CTA's sorted bottom 32 go to every CTA.
    if (!skip) lst[warp * 32 + lane] = warp_sort32(mykey, lane);
    __syncthreads();
    if (!skip && (warp & 1) == 0)
      lst[warp * 32 + lane] = warp_merge_low32(lst[warp * 32 + lane], lst[(warp + 1) * 32 + lane], lane);
    __syncthreads();
    if (!skip && (warp & 3) == 0)
      lst[warp * 32 + lane] = warp_merge_low32(lst[warp * 32 + lane], lst[(warp + 2) * 32 + lane], lane);
    __syncthreads();
    if (!skip && warp == 0) {
      const unsigned long long mine = warp_merge_low32(lst[lane], lst[4 * 32 + lane], lane);
      const uint32_t local = smem_u32(&s.cand_recv[c * 32 + lane]);
      for (int dst = 0; dst < C; ++dst) st_cluster_u64(mapa(local, dst), mine);
    }
  } else {
    // Many evictions (the first compression after a long prefill).  Each warp sorts its 32
    // keys; each key then takes its place in the CTA's sorted list by counting the smaller
    // keys of the other warps' sorted runs (binary search), so the cross-warp part of the sort
    // costs one CTA barrier.  After a cluster barrier thread i takes key i of its CTA's sorted
    // list: i keys of its own CTA lie below it, and the smaller keys of every other CTA are
    // counted by binary search in local copies of their sorted lists (one coalesced remote
    // load per thread and list, all issued at once, kSelBufs lists searched per round).  The
    // evicted keys of the CTA are the prefix of its sorted list whose ranks are below E.
    constexpr int kWarps = kThreads / 32;
    constexpr int NB = kSelBufs<MAXC>;
    unsigned long long* const runs = s.u1.sel.copy[0];
    unsigned long long xs = 0ull;
    if (!skip) {  // uniform over the cluster
      xs = warp_sort32(mykey, lane);
      runs[tid] = xs;
    }
    __syncthreads();
    if (!skip) {
      int pw[kWarps - 1];
#pragma unroll
      for (int i = 0; i < kWarps - 1; ++i) pw[i] = 0;
#pragma unroll
      for (int step = 16; step > 0; step >>= 1)
#pragma unroll
        for (int i = 0; i < kWarps - 1; ++i)
          if (runs[((warp + 1 + i) % kWarps) * 32 + pw[i] + step - 1] < xs) pw[i] += step;
      int pos = lane;
#pragma unroll
      for (int i = 0; i < kWarps - 1; ++i)
        pos += pw[i] + (runs[((warp + 1 + i) % kWarps) * 32 + pw[i]] < xs ? 1 : 0);
      lst[pos] = xs;
    }
    cluster_sync();  // every CTA's sorted list is complete (and this CTA's runs are read)
    bool ev_sorted = false;
    if (!skip) {
      const unsigned long long x = lst[tid];
      unsigned long long rk[MAXC - 1];  // the other CTAs' lists, starting after this one
      const uint32_t mine = smem_u32(&lst[tid]);
#pragma unroll
      for (int i = 0; i < MAXC - 1; ++i) {
        int cc = c + 1 + i;
        if (cc >= C) cc -= C;
        rk[i] = i < C - 1 ? ld_cluster_u64(mapa(mine, cc)) : 0ull;
      }
      int rank = tid;
#pragma unroll
      for (int r0 = 0; r0 < MAXC - 1; r0 += NB) {
        if (r0 >= C - 1) break;  // C is uniform over the cluster
        const int nr = min(NB, C - 1 - r0);
#pragma unroll
        for (int i = 0; i < NB; ++i)
          if (r0 + i < MAXC - 1 && i < nr) sel_buf(s, i)[tid] = rk[r0 + i];
        __syncthreads();
        // keys below x in each list: the halving steps reach 255 at most, the last compare
        // counts the list's last key
        int p[NB];
#pragma unroll
        for (int i = 0; i < NB; ++i) p[i] = 0;
#pragma unroll
        for (int step = kKeysPerCta / 2; step > 0; step >>= 1)
#pragma unroll
          for (int i = 0; i < NB; ++i)
            if (r0 + i < MAXC - 1 && i < nr && sel_buf(s, i)[p[i] + step - 1] < x) p[i] += step;
#pragma unroll
        for (int i = 0; i < NB; ++i)
          if (r0 + i < MAXC - 1 && i < nr) rank += p[i] + (sel_buf(s, i)[p[i]] < x ? 1 : 0);
        if (r0 + NB < C - 1) __syncthreads();  // the next round overwrites the copies
      }
      ev_sorted = rank < E;
    }
    // ranks grow along the sorted list, so this CTA's evicted keys are its first m keys
    const int m = __syncthreads_count(!skip && ev_sorted);
    if (!skip) evicted = key_valid && (m >= kKeysPerCta || mykey < lst[m]);
    const int kept_cta = __syncthreads_count(!skip && key_valid && !evicted);
    if (!skip && tid == 0) {
      const uint32_t local = smem_u32(&s.kept_recv[c]);
      for (int dst = 0; dst < C; ++dst) st_cluster_u32(mapa(local, dst), static_cast<uint32_t>(kept_cta));
    }
  }
  if (!skip && tid == 0) {
    bool vok = true;
    if (v_pending) {
      vok = mbar_wait_bounded(&s.bar_v, ph_v, kWaitNs);  // staged V rows have landed
      if (vok) {
        ph_v ^= 1;
        v_pending = false;
      }
    }
    ok = ok && vok;
    const uint32_t local = smem_u32(&s.status_recv[c]);
    for (int dst = 0; dst < C; ++dst) st_cluster_u32(mapa(local, dst), (fail || !ok) ? 1u : 0u);
  }
  if (c == 0 && tid == 0) {  // the next unit reaches every CTA with this barrier, skipped or not
    const uint32_t nl = smem_u32(&s.next_unit[iter & 1]);
    for (int dst = 0; dst < C; ++dst) st_cluster_u32(mapa(nl, dst), static_cast<uint32_t>(next_fetch));
  }
  cluster_sync();  // #2: candidates, statuses and every read of every CTA of the unit are done
  const int next_unit = s.next_unit[iter & 1];

  bool any_fail = false;
  if (!skip) {
    for (int cc = 0; cc < C; ++cc) any_fail |= s.status_recv[cc] != 0;
    int j = -1;  // destination slot of this thread's key if kept
    if (E <= 32) {
      // cluster level: merge the C sorted lists (missing lists count as +inf), identically in
      // every CTA; the first E keys of the result are evicted.  Scratch in u0: the u1 buffers
      // may already receive the next unit's row statistics.
      // Pairwise tree: level 1 merges the MAXC lists into MAXC/2, ..., down to 2 lists, which
      // warp 0 merges into the final one.
      static_assert(MAXC == 8 || MAXC == 16, "merge tree of 8 or 16 lists");
      unsigned long long* lvl = s.u0.lists;  // [MAXC/2][32], then [MAXC/4][32], ...
      if (warp < MAXC / 2) {
        const unsigned long long x0 = (2 * warp < C) ? s.cand_recv[(2 * warp) * 32 + lane] : ~0ull;
        const unsigned long long x1 = (2 * warp + 1 < C) ? s.cand_recv[(2 * warp + 1) * 32 + lane] : ~0ull;
        lvl[warp * 32 + lane] = warp_merge_low32(x0, x1, lane);
      }
      __syncthreads();
      if constexpr (MAXC >= 16) {  // 8 lists -> 4
        unsigned long long* const nxt = lvl + 8 * 32;
        if (warp < 4)
          nxt[warp * 32 + lane] = warp_merge_low32(lvl[(2 * warp) * 32 + lane], lvl[(2 * warp + 1) * 32 + lane], lane);
        __syncthreads();
        lvl = nxt;
      }
      {  // 4 lists -> 2
        unsigned long long* const nxt = lvl + 4 * 32;
        if (warp < 2)
          nxt[warp * 32 + lane] = warp_merge_low32(lvl[(2 * warp) * 32 + lane], lvl[(2 * warp + 1) * 32 + lane], lane);
        __syncthreads();
        lvl = nxt;
      }
      if (warp == 0) {
        const unsigned long long fin = warp_merge_low32(lvl[lane], lvl[32 + lane], lane);
        if (lane < E) s.evict_pos[lane] = static_cast<int>(0xFFFFFFFFu - static_cast<uint32_t>(fin & 0xFFFFFFFFu));
      }
      __syncthreads();
      // j = t - #(evicted before t)
      if (key_valid) {
        int shift = 0;
        for (int e = 0; e < E; ++e) {
          const int p = s.evict_pos[e];
          shift += (p < kt) ? 1 : 0;
          evicted |= (p == kt);
        }
        if (!evicted) j = kt - shift;
      }
    } else {
      // j = kept keys of the earlier CTAs + kept keys before t in this CTA
      const bool kept = key_valid && !evicted;
      const unsigned ball = __ballot_sync(0xffffffffu, kept);
      if (lane == 0) s.warp_kept[warp] = __popc(ball);
      __syncthreads();
      int before = 0;
      for (int cc = 0; cc < c; ++cc) before += s.kept_recv[cc];
      for (int ww = 0; ww < warp; ++ww) before += s.warp_kept[ww];
      if (kept) j = before + __popc(ball & ((1u << lane) - 1));
    }
    if (j >= 0) g_in = a.decay * g_in + attn;  // global-score update of the kept key
    if (key_valid && a.dbg_keep)
      a.dbg_keep[((static_cast<int64_t>(r) * a.layers + layer) * a.Hkv + h) * La + kt] = j >= 0 ? 1 : 0;
    const bool moved = j >= 0 && (s.src_tab[kt >> bs] != s.dst_tab[j >> bs] || (kt & bm) != (j & bm));
    s.dst_of[tid] = moved ? j : -1;
    __syncthreads();

    if (!any_fail) {
      // K from shared memory (swizzled rows), V from the staging area or registers.  Warp w
      // writes rows 16w .. 16w + 15 and 128 + 16w .. 128 + 16w + 15.
      const int ch = lane % cpr, half = ch >> 3, c8 = ch & 7;
#pragma unroll
      for (int it = 0; it < 8; ++it) {
        if (it * rpi >= 16) break;
        const int sub = it * rpi + lane / cpr;
#pragma unroll
        for (int part = 0; part < 2; ++part) {
          const int row = part * 128 + warp * 16 + sub;
          if (row >= nk) continue;
          const int jj = s.dst_of[row];
          if (jj < 0) continue;
          const uint4 kv = *reinterpret_cast<const uint4*>(&s.K[half][row * 128 + ((c8 ^ (row & 7)) << 4)]);
          const uint4 vv = part == 0 ? *reinterpret_cast<const uint4*>(vstage + row * a.row_bytes + ch * 16) : vreg[it];
          uint8_t* dk = head_base + row_off_bytes(a, s.dst_tab[jj >> bs], 0, jj & bm) + ch * 16;
          *reinterpret_cast<uint4*>(dk) = kv;
          *reinterpret_cast<uint4*>(dk + a.kv_bytes) = vv;
        }
      }
      float* G = a.gscores + ((static_cast<int64_t>(slot) * a.layers + layer) * a.Hkv + h) * La;
      if (j >= 0) G[j] = g_in;
      if (kt >= k_r && kt < L) G[kt] = 0.0f;  // slots past the k survivors
    }
  }
  if (!skip && any_fail && tid == 0 && c == 0) record_error(a.err, ZP_ERR_TIMEOUT);
  // copies a skipped or failed unit issued and never saw complete: wait (bounded) before the
  // shared memory is reused
  if (tid == 0) {
    if (tma_pending && mbar_wait_bounded(&s.bar_tma, ph_tma, kWaitNs)) ph_tma ^= 1;
    if (v_pending && mbar_wait_bounded(&s.bar_v, ph_v, kWaitNs)) ph_v ^= 1;
  }
  // every generic read of K / the staging area and every TMEM load of this unit precedes the
  // next unit's TMA and MMAs
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  unit = next_unit;
  }  // unit loop

  if (warp == 0) tmem_dealloc(tbase, kTmemCols);
}

// Workspace header of the fused form: the error word (int 0), the unit counter of a single
// launch (int 1), one unit counter per length group (ints 16 + C) and one (first position,
// request count) pair per group (ints 48 + 2C); the grouped request order follows it.
constexpr int kWsGroupCounters = 16;
constexpr int kWsGroups = 48;
constexpr size_t kWsHeaderBytes = 512;
static_assert(kWsGroups * 4 >= (kWsGroupCounters + kMaxCluster + 1) * 4, "header fields overlap");
static_assert((kWsGroups + 2 * (kMaxCluster + 1)) * 4 <= static_cast<int>(kWsHeaderBytes), "header too small");

// Groups the requests by the CTAs their length needs (C_r = ceil(L_r / 256)), so that each
// group runs in clusters of its own size and no CTA waits through a unit with no keys.
// A request whose length cannot be valid (L_r <= k_lo or L_r > L) goes to the largest group,
// whose kernel reports it.  One CTA; thread i takes a contiguous run of requests, so the
// order inside a group is the request order.
constexpr int kPlanThreads = 256;
constexpr int kGroups = kMaxCluster + 1;  // group c holds requests of c CTAs (c = 0 unused)
__global__ void __launch_bounds__(kPlanThreads) group_by_length_kernel(const int32_t* seq_len, int R, int L, int k_lo,
                                                                       int c_max, int32_t* ws) {
  __shared__ int cnt[kGroups][kPlanThreads];  // per (group, thread): count, then first position
  __shared__ int total[kGroups], first[kGroups];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int per = (R + kPlanThreads - 1) / kPlanThreads;
  const int r0 = min(R, tid * per), r1 = min(R, r0 + per);
  for (int c = 0; c < kGroups; ++c) cnt[c][tid] = 0;
  auto group_of = [&](int r) {
    const int Lr = seq_len[r];
    return (Lr > k_lo && Lr <= L) ? (Lr + kKeysPerCta - 1) / kKeysPerCta : c_max;
  };
  for (int r = r0; r < r1; ++r) ++cnt[group_of(r)][tid];
  __syncthreads();
  // exclusive scan over the threads, one group per warp at a time: lane l takes the 8
  // consecutive threads 8l .. 8l + 7
  constexpr int kPerLane = kPlanThreads / 32;
  for (int c = warp; c < kGroups; c += kPlanThreads / 32) {
    int v[kPerLane], sum = 0;
#pragma unroll
    for (int j = 0; j < kPerLane; ++j) {
      v[j] = cnt[c][lane * kPerLane + j];
      sum += v[j];
    }
    int incl = sum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    int run = incl - sum;
#pragma unroll
    for (int j = 0; j < kPerLane; ++j) {
      cnt[c][lane * kPerLane + j] = run;
      run += v[j];
    }
    if (lane == 31) total[c] = incl;
  }
  __syncthreads();
  if (tid < kGroups) {
    int base = 0;
    for (int c = 0; c < tid; ++c) base += total[c];
    ws[kWsGroups + 2 * tid] = base;
    ws[kWsGroups + 2 * tid + 1] = total[tid];
    ws[kWsGroupCounters + tid] = 0;
    first[tid] = base;
  }
  __syncthreads();
  int32_t* order = ws + kWsHeaderBytes / 4;
  for (int r = r0; r < r1; ++r) {
    const int c = group_of(r);
    order[first[c] + cnt[c][tid]++] = r;
  }
}

// Cluster sizes of one call: requests whose lengths may need different cluster sizes (a launch
// length above n_max*b, or per-request budgets) are grouped by length on the device, and each
// group runs in a launch of its own cluster size c in [c_lo, C]; otherwise (c_lo == C) one
// launch covers every request.  k_lo is the smallest budget a request may have.
struct ClusterPlan {
  int C, c_lo, k_lo;
};
ClusterPlan cluster_plan(int L, int k, int b, bool per_request_budgets) {
  ClusterPlan q;
  q.C = (L + kKeysPerCta - 1) / kKeysPerCta;
  q.k_lo = per_request_budgets ? b : k;
  q.c_lo = std::min(q.C, (q.k_lo + 1 + kKeysPerCta - 1) / kKeysPerCta);
  return q;
}

}  // namespace

template <int MAXC>
size_t compress_smem_bytes() { return sizeof(SmemT<MAXC>) + 1024; }

// Launches the persistent clusters of compress_kernel<MAXC> (C <= MAXC CTAs each).
template <int MAXC>
zp_status launch_compress(const CUtensorMap& tmK, const CUtensorMap& tmQ, const CompressArgs& a, int C,
                          int64_t num_units, cudaStream_t st) {
  const size_t smem = compress_smem_bytes<MAXC>();
  static PerDeviceInit attrs;
  const cudaError_t attr_err = attrs.run([&] {
    cudaError_t e = cudaFuncSetAttribute(compress_kernel<MAXC>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e == cudaSuccess && MAXC > 8)
      e = cudaFuncSetAttribute(compress_kernel<MAXC>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    return e;
  });
  if (attr_err != cudaSuccess) return ZP_ERR_CUDA;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(C, 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = C;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  // as many clusters as are co-resident (persistent), never more than there are units
  static std::mutex occ_mu;
  static int occ_cache[64][MAXC + 1] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return ZP_ERR_CUDA;
  int max_clusters = 0;
  {
    std::lock_guard<std::mutex> lock(occ_mu);
    if (dev >= 0 && dev < 64 && occ_cache[dev][C] > 0) {
      max_clusters = occ_cache[dev][C];
    } else {
      if (cudaOccupancyMaxActiveClusters(&max_clusters, compress_kernel<MAXC>, &cfg) != cudaSuccess ||
          max_clusters <= 0)
        max_clusters = 1;
      if (dev >= 0 && dev < 64) occ_cache[dev][C] = max_clusters;
    }
  }
  // Units are handed out dynamically, so launching more clusters than can be resident only
  // leaves the late ones an empty queue; MAXC <= 8 fits two CTAs per SM, 16 one.
  const int per_sm = MAXC <= 8 ? 2 : 1;
  const int64_t want = std::max<int64_t>(max_clusters, (per_sm * static_cast<int64_t>(num_sms())) / C);
  const int64_t clusters = std::max<int64_t>(1, std::min<int64_t>(num_units, want));
  cfg.gridDim = dim3(static_cast<unsigned>(C * clusters), 1, 1);
  if (cudaLaunchKernelEx(&cfg, compress_kernel<MAXC>, tmK, tmQ, a) != cudaSuccess) return ZP_ERR_CUDA;
  return ZP_OK;
}

}  // namespace zp

using namespace zp;

// The error word and the unit counters, then the grouped request order of the fused form, or,
// for sequences beyond one cluster (L > 4096), the scratch of the multi-pass form.
extern "C" size_t zp_compress_workspace_size(const zp_params* p, int32_t num_requests, int32_t max_seq_len) {
  if (!p || num_requests < 0) return 0;
  const int64_t L = max_seq_len > 0 ? max_seq_len : static_cast<int64_t>(p->n_max) * p->block_size;
  if (L <= static_cast<int64_t>(kMaxCluster) * kKeysPerCta)
    return kWsHeaderBytes + ((static_cast<size_t>(num_requests) * 4 + 255) & ~size_t(255));
  return 256 + compress_long_scratch_bytes(static_cast<int64_t>(num_requests) * p->num_layers * p->num_kv_heads,
                                           static_cast<int>(L));
}

namespace {
// The compression call; stall_ns != 0 only from the test hook (multi-pass form).
zp_status compress_call(const zp_kv_pool* pool, const int32_t* block_tables, const zp_seq_meta* meta,
                        const uint16_t* obs_q, int32_t num_qslots, float* global_scores, const zp_params* p,
                        const zp_debug* dbg, void* workspace, size_t workspace_bytes, zp_stream stream,
                        uint64_t stall_ns) {
  if (!pool || !meta || !obs_q || !global_scores || !p || !workspace) return ZP_ERR_INVALID_ARG;
  if (!pool->base || pool->num_blocks <= 0) return ZP_ERR_INVALID_ARG;
  // with no request the per-request arrays may be empty (NULL)
  if (meta->num_requests > 0 && (!block_tables || !meta->seq_len || !meta->qslot || !meta->dst_tables))
    return ZP_ERR_INVALID_ARG;
  if (workspace_bytes < zp_compress_workspace_size(p, meta->num_requests, meta->max_seq_len) ||
      !aligned(workspace, 256))
    return ZP_ERR_INVALID_ARG;
  const int layers = p->num_layers, Hq = p->num_q_heads, Hkv = p->num_kv_heads, d = p->head_dim,
            b = p->block_size, n_max = p->n_max, w = p->window, R = meta->num_requests;
  if (layers <= 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0 || R < 0 || num_qslots <= 0) return ZP_ERR_INVALID_ARG;
  if (n_max < 2 || meta->max_blocks < n_max || w < 1) return ZP_ERR_INVALID_ARG;
  // the call's layers (all of them unless a range is given)
  const int layer_begin = meta->layer_count > 0 ? meta->layer_begin : 0;
  const int nl = meta->layer_count > 0 ? meta->layer_count : layers;
  if (meta->layer_count < 0 || (meta->layer_count == 0 && meta->layer_begin != 0) || layer_begin < 0 ||
      layer_begin + nl > layers)
    return ZP_ERR_INVALID_ARG;
  const int k = (n_max - 1) * b, Gq = Hq / Hkv, Rw = w * Gq;
  // launch length: the longest request of the call (n_max*b unless the caller says more)
  const int L = meta->max_seq_len > 0 ? meta->max_seq_len : n_max * b;
  if (w > k || L <= k) return ZP_ERR_INVALID_ARG;
  if (meta->max_blocks < (L + b - 1) / b) return ZP_ERR_INVALID_ARG;
  if (d != 64 && d != 128) return ZP_ERR_UNSUPPORTED;
  if (b != 16 && b != 32) return ZP_ERR_UNSUPPORTED;
  // one cluster of up to 16 CTAs covers L <= 4096; longer sequences (to 16384) take the
  // multi-pass form
  // (n_max <= L/b + 1 <= max_table(16) whenever one cluster covers L)
  if (Rw > kRows || L > 16384) return ZP_ERR_UNSUPPORTED;
  if (Gq > 256 || w > 256) return ZP_ERR_UNSUPPORTED;
  if (!aligned(pool->base, 16) || !aligned(obs_q, 16)) return ZP_ERR_INVALID_ARG;
  if (static_cast<int64_t>(layers) * pool->num_blocks >= (int64_t(1) << 31)) return ZP_ERR_UNSUPPORTED;
  if (static_cast<int64_t>(R) * layers * Hkv >= (int64_t(1) << 31)) return ZP_ERR_UNSUPPORTED;
  if (static_cast<int64_t>(num_qslots) * layers * w >= (int64_t(1) << 31)) return ZP_ERR_UNSUPPORTED;

  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (cudaMemsetAsync(workspace, 0, 8, st) != cudaSuccess) return ZP_ERR_CUDA;  // error word, unit counter
  if (R == 0) return ZP_OK;

  CUtensorMap tmK, tmQ;
  // K/V pool as {d, 2*Hkv*b rows per (layer, block), layers*num_blocks}; box = one block's
  // b rows of one head, 64 columns.
  if (!encode_tmap_3d_bf16(&tmK, pool->base, d, static_cast<uint64_t>(2) * Hkv * b,
                           static_cast<uint64_t>(layers) * pool->num_blocks, static_cast<uint64_t>(d) * 2,
                           static_cast<uint64_t>(2) * Hkv * b * d * 2, 64, b, 1))
    return ZP_ERR_CUDA;
  // window queries as {d, Hq, slots*layers*w}; box = the G_q heads of one kv head x w rows.
  if (!encode_tmap_3d_bf16(&tmQ, obs_q, d, Hq, static_cast<uint64_t>(num_qslots) * layers * w,
                           static_cast<uint64_t>(d) * 2, static_cast<uint64_t>(Hq) * d * 2, 64, Gq, w))
    return ZP_ERR_CUDA;

  CompressArgs a{};
  a.pool = static_cast<uint8_t*>(pool->base);
  a.num_blocks = pool->num_blocks;
  a.block_tables = block_tables;
  a.dst_tables = meta->dst_tables;
  a.seq_len = meta->seq_len;
  a.qslot = meta->qslot;
  a.n_max_req = meta->n_max_per_req;
  a.gscores = global_scores;
  a.err = static_cast<int32_t*>(workspace);
  a.work = static_cast<int32_t*>(workspace) + 1;
  if (dbg) {
    a.dbg_attn = dbg->attn;
    a.dbg_redund = dbg->redund;
    a.dbg_score = dbg->score;
    a.dbg_keep = dbg->keep;
  }
  a.R = R;
  a.layers = layers;
  a.layer0 = layer_begin;
  a.nl = nl;
  a.Hq = Hq;
  a.Hkv = Hkv;
  a.d = d;
  a.b = b;
  a.n_max = n_max;
  a.w = w;
  a.Gq = Gq;
  a.Rw = Rw;
  a.L = L;
  a.k = k;
  a.max_blocks = meta->max_blocks;
  a.num_qslots = num_qslots;
  a.alpha = p->alpha;
  a.beta = p->beta;
  a.decay = p->decay;
  a.sl2 = p->scale * 1.4426950408889634f;
  a.inv_rw = 1.0f / static_cast<float>(Rw);
  a.row_bytes = static_cast<uint32_t>(d) * 2;
  a.b_shift = (b == 16) ? 4 : 5;
  a.kv_bytes = static_cast<uint32_t>(Hkv) * b * a.row_bytes;
  a.block_bytes = 2 * a.kv_bytes;
  a.protect_window = p->protect_window;
  a.causal = p->causal;
  a.stall_ns = stall_ns;

  const ClusterPlan plan = cluster_plan(L, k, b, meta->n_max_per_req != nullptr);
  const int C = plan.C, c_lo = plan.c_lo;
  if (C > kMaxCluster) return launch_compress_long(tmK, tmQ, a, static_cast<uint8_t*>(workspace) + 256, st);
  const int64_t num_units = static_cast<int64_t>(R) * nl * Hkv;
  a.Lc = L;
  if (c_lo == C) return C <= 8 ? launch_compress<8>(tmK, tmQ, a, C, num_units, st)
                               : launch_compress<16>(tmK, tmQ, a, C, num_units, st);
  int32_t* ws = static_cast<int32_t*>(workspace);
  group_by_length_kernel<<<1, kPlanThreads, 0, st>>>(meta->seq_len, R, L, plan.k_lo, C, ws);
  if (cudaGetLastError() != cudaSuccess) return ZP_ERR_CUDA;
  a.req_order = ws + kWsHeaderBytes / 4;
  for (int c = c_lo; c <= C; ++c) {
    CompressArgs ac = a;
    ac.Lc = std::min(L, c * kKeysPerCta);
    ac.work = ws + kWsGroupCounters + c;
    ac.bucket = ws + kWsGroups + 2 * c;
    const zp_status stc = c <= 8 ? launch_compress<8>(tmK, tmQ, ac, c, num_units, st)
                                 : launch_compress<16>(tmK, tmQ, ac, c, num_units, st);
    if (stc != ZP_OK) return stc;
  }
  return ZP_OK;
}
}  // namespace

extern "C" zp_status zp_compress(const zp_kv_pool* pool, const int32_t* block_tables, const zp_seq_meta* meta,
                                 const uint16_t* obs_q, int32_t num_qslots, float* global_scores,
                                 const zp_params* p, const zp_debug* dbg, void* workspace,
                                 size_t workspace_bytes, zp_stream stream) {
  zp::NvtxRange nvtx_range("zp_compress");
  return compress_call(pool, block_tables, meta, obs_q, num_qslots, global_scores, p, dbg, workspace, workspace_bytes,
                       stream, 0);
}

extern "C" zp_status zp_test_compress_stalled(const zp_kv_pool* pool, const int32_t* block_tables,
                                              const zp_seq_meta* meta, const uint16_t* obs_q, int32_t num_qslots,
                                              float* global_scores, const zp_params* p, void* workspace,
                                              size_t workspace_bytes, int64_t stall_limit_ns, zp_stream stream) {
  if (stall_limit_ns < 1 || stall_limit_ns > 1000000000) return ZP_ERR_INVALID_ARG;
  // the multi-pass form only: its CTAs exchange nothing, so a wait that gives up stays local
  if (!meta || !p || meta->max_seq_len <= kMaxCluster * kKeysPerCta) return ZP_ERR_INVALID_ARG;
  return compress_call(pool, block_tables, meta, obs_q, num_qslots, global_scores, p, nullptr, workspace,
                       workspace_bytes, stream, static_cast<uint64_t>(stall_limit_ns));
}

extern "C" int32_t zp_compress_kernel_launches(const zp_params* p, int32_t max_seq_len, int32_t per_request_budgets) {
  if (!p || p->n_max < 2 || (p->block_size != 16 && p->block_size != 32)) return 0;
  const int b = p->block_size, k = (p->n_max - 1) * b;
  const int L = max_seq_len > 0 ? max_seq_len : p->n_max * b;
  if (L <= k || L > 16384) return 0;
  const ClusterPlan plan = cluster_plan(L, k, b, per_request_budgets != 0);
  if (plan.C > kMaxCluster) return 4;  // statistics, scores, selection, compaction
  return plan.c_lo == plan.C ? 1 : 1 + (plan.C - plan.c_lo + 1);
}
