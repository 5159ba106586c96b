// zp_decode.cu — paged decode attention over the (compacted) KV cache, sm_103a.
//
// The consumer of the compression pass: requests that are not compressing keep decoding
// while compression runs on a side stream (Zipage summaries on gist.science: zh §2.1
// asynchronous compression and decoding, zh §2.3 PagedAttention/FlashAttention integration,
// fr §2.D).  One new token per request and one layer per launch:
//   out[r][qh] = sum_t softmax_t(scale * <q[r][qh], k_t>) v_t,  t < seq_lens[r],
// with k_t, v_t of kv head qh / G_q read through block_tables[r].
//
// Split-KV flash decoding on the warp-level tensor cores.  Grid (split of 32 blocks, kv head,
// request); each CTA of 4 warps walks its split's blocks (warp w takes blocks w, w+4, ...).  A
// warp streams its blocks in chunks of 16 rows through two shared-memory stages: TMA brings a
// chunk's K rows and V rows (128-byte swizzle, completing on the stage's mbarrier) while the
// warp computes on the other stage.  The G_q query heads of the kv head are the rows of an
// m16n8k16 MMA (padded to 16): S = Q K^T from ldmatrix fragments of K, an online softmax per
// row in the log2 domain, then O += P V with V fragments from ldmatrix.trans.  P enters the
// MMA as a bf16 high part plus a bf16 remainder, which keeps about 16 bits of it; the exp-sum
// uses the fp32 values.  Warps are merged at the end; with more than one split the
// (max, sum, acc) partials go to the workspace and a second kernel merges the splits.
#include "zp_internal.h"
#include "zp_ptx.cuh"

#include <mutex>

namespace zp {
namespace {

constexpr int kWarps = 4;
constexpr int kThreads = kWarps * 32;
// KV blocks per CTA (a split): 32, 64 or 128 (<= 32 * kWarps: a lane holds each block id of
// its warp), chosen per launch; workspaces are sized for the smallest
constexpr int kMinBlocksPerSplit = 32;
constexpr int kMaxBlocksPerSplit = 32 * kWarps;
constexpr int kChunkRows = 16;       // rows per bulk-copied K (and V) chunk: b = 16 or 32
constexpr uint64_t kWaitNsD = 2000000000ull;

struct DecodeArgs {
  const uint8_t* pool;
  int64_t num_blocks;
  const uint16_t* q;
  const int32_t* tables;
  const int32_t* seq_lens;
  uint16_t* out;
  float* part;  // [B][Hq][max_splits][d + 2]
  int32_t* err;
  int B, layer, Hq, Hkv, d, b, Gq, max_blocks, max_splits;
  int bps;    // blocks per split of this launch
  float sl2;  // scale * log2(e)
  // test hook of the bounded waits, 0 in normal calls: before its first chunk every warp also
  // waits this long on a barrier that nothing completes, so the wait runs out
  uint64_t stall_ns;
};

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}


__device__ __forceinline__ uint16_t f2bf16(float f) {
  // round to nearest even; NaN stays NaN
  uint32_t u = __float_as_uint(f);
  if ((u & 0x7FFFFFFFu) > 0x7F800000u) return static_cast<uint16_t>((u >> 16) | 0x40u);
  u += 0x7FFFu + ((u >> 16) & 1u);
  return static_cast<uint16_t>(u >> 16);
}

// Packs two floats into a bf16x2 register (lo in the low half), rounding to nearest even.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}
__device__ __forceinline__ float bf16x2_lo(uint32_t u) { return __uint_as_float(u << 16); }
__device__ __forceinline__ float bf16x2_hi(uint32_t u) { return __uint_as_float(u & 0xFFFF0000u); }

// Byte offset, inside a (16-row, D-column) chunk stored as [d/64 half][16 rows][128 B] with the
// 128-byte swizzle that TMA applies, of 16-byte column group `cg` (0 .. D/8-1) of row `row`.
template <int D>
__device__ __forceinline__ uint32_t swz_off(int row, int cg) {
  return static_cast<uint32_t>((cg >> 3) * (kChunkRows * 128) + row * 128 + (((cg & 7) ^ (row & 7)) << 4));
}

template <int D, int G>
__global__ void __launch_bounds__(kThreads) decode_kernel(const __grid_constant__ CUtensorMap tm, const DecodeArgs a) {
  constexpr int NH = D / 64;                   // 64-column halves
  constexpr int kChunkBytes = kChunkRows * D * 2;
  constexpr int NT = D / 8;                    // n8 tiles of the output row
  __shared__ float sm_m[kWarps][G], sm_l[kWarps][G];
  __shared__ float sm_acc[kWarps][G][D];
  __shared__ int sm_bad;
  __shared__ __align__(8) uint64_t sm_bar[kWarps][2];
  __shared__ __align__(8) uint64_t sm_never;  // test hook: no thread or copy ever arrives on it
  // per warp, two stages of (K, V) chunks of kChunkRows rows in the TMA's 128-byte swizzle
  // (dynamic shared memory, 1024-byte aligned below)
  extern __shared__ uint8_t dyn_smem[];
  uint8_t* const kv_base =
      reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(dyn_smem) + 1023) & ~uintptr_t(1023));

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int split = blockIdx.x, h = blockIdx.y, r = blockIdx.z;
  const int fr = lane >> 2, q = lane & 3;      // mma fragment row (query head) and column pair
  const int seq = a.seq_lens[r];
  const int b = a.b;
  const int cpb = b / kChunkRows;              // chunks per block
  const int nblk = (seq + b - 1) / b;
  const int blk0 = split * a.bps;
  const int blk1 = min(nblk, blk0 + a.bps);

  if (tid == 0) {
    sm_bad = (seq < 1 || seq > a.max_blocks * b) ? 1 : 0;
    mbar_init(&sm_never, 1);
  }
  if (lane == 0) {
    mbar_init(&sm_bar[warp][0], 1);
    mbar_init(&sm_bar[warp][1], 1);
    fence_mbar_init();
  }
  if (tid == 0) prefetch_tensormap(&tm);
  __syncthreads();
  if (sm_bad) {
    if (tid == 0 && split == 0 && h == 0) atomicCAS(a.err, 0, ZP_ERR_BAD_TABLE);
    return;
  }
  if (blk0 >= nblk) return;  // this split has no work (uniform over the CTA)

  // Q as mma A fragments (rows = the G query heads, padded to 16 with zeros): per k-step of 16
  // columns, qa[ks][0] holds row fr, columns 16ks + 2q, +1 and qa[ks][1] columns 16ks + 8 + 2q, +1.
  uint32_t qa[D / 16][2];
#pragma unroll
  for (int ks = 0; ks < D / 16; ++ks) {
    qa[ks][0] = qa[ks][1] = 0u;
    if (fr < G) {
      const uint32_t* qrow =
          reinterpret_cast<const uint32_t*>(a.q + (static_cast<int64_t>(r) * a.Hq + h * G + fr) * D);
      qa[ks][0] = qrow[(16 * ks + 2 * q) >> 1];
      qa[ks][1] = qrow[(16 * ks + 8 + 2 * q) >> 1];
    }
  }
  // running max (log2 domain), this thread's share of the exp-sum, and the output row fr at
  // columns 8nt + 2q, +1 (o[nt][2], o[nt][3] belong to padding rows)
  float m = -INFINITY, l = 0.0f;
  float o[NT][4];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) o[nt][0] = o[nt][1] = o[nt][2] = o[nt][3] = 0.0f;

  // This warp's blocks are blk0 + warp + kWarps*i (i < nb); lane i holds the physical id of
  // the i-th one (a split's blocks / kWarps <= 32), so issuing a copy needs no global load.
  const int nb = (blk1 - blk0 - warp + kWarps - 1) / kWarps;  // may be <= 0
  const int32_t* table = a.tables + static_cast<int64_t>(r) * a.max_blocks;
  const int my_phys = (lane < nb) ? table[blk0 + warp + kWarps * lane] : 0;
  const bool my_bad = lane < nb && (my_phys < 0 || my_phys >= a.num_blocks);
  const bool bad = __any_sync(0xffffffffu, my_bad);
  const int nch = bad ? 0 : nb * cpb;  // chunks of this warp (none if a block id is bad)
  uint8_t* const wbuf = kv_base + warp * (2 * 2 * kChunkBytes);  // [stage][K|V][chunk]
  // chunk c of this warp: rows [(c % cpb) * kChunkRows, +kChunkRows) of its (c / cpb)-th block;
  // in the pool viewed as {d, 2*Hkv*b rows, layers*blocks}, K rows of head h start at h*b and
  // V rows at (Hkv + h)*b
  auto issue = [&](int c, int st) {
    const int phys = __shfl_sync(0xffffffffu, my_phys, c / cpb);
    if (lane == 0) {
      uint64_t* bar = &sm_bar[warp][st];
      const int row = h * b + (c % cpb) * kChunkRows, z = a.layer * static_cast<int>(a.num_blocks) + phys;
      mbar_arrive_expect_tx(bar, 2u * kChunkBytes);
#pragma unroll
      for (int hd = 0; hd < NH; ++hd) {
        tma_load_3d(wbuf + (st * 2 + 0) * kChunkBytes + hd * kChunkRows * 128, &tm, bar, hd * 64, row, z);
        tma_load_3d(wbuf + (st * 2 + 1) * kChunkBytes + hd * kChunkRows * 128, &tm, bar, hd * 64,
                    a.Hkv * b + row, z);
      }
    }
  };
  // ldmatrix rows: lanes 0-7 / 8-15 / 16-23 / 24-31 address matrices 0..3 = (rows 0-7, group j),
  // (rows 8-15, group j), (rows 0-7, group j+1), (rows 8-15, group j+1)
  const int lrow = (lane & 7) + ((lane >> 3) & 1) * 8, lgrp = lane >> 4;
  uint32_t ph = 0;  // phase bit of each stage's barrier
  bool ok = true;
  int c = 0;
  if (nch > 0) issue(0, 0);
  if (nch > 1) issue(1, 1);
  for (; c < nch; ++c) {
    const int st = c & 1;
    bool w = true;
    if (lane == 0) {
      if (a.stall_ns != 0 && c == 0) w = mbar_wait_bounded(&sm_never, 0u, a.stall_ns);  // runs out
      if (w) w = mbar_wait_bounded(&sm_bar[warp][st], (ph >> st) & 1u, kWaitNsD);
    }
    w = __shfl_sync(0xffffffffu, w, 0);
    if (!w) {
      ok = false;
      break;
    }
    ph ^= 1u << st;
    const uint32_t kbuf = smem_u32(wbuf + (st * 2 + 0) * kChunkBytes);
    const uint32_t vbuf = smem_u32(wbuf + (st * 2 + 1) * kChunkBytes);
    const int tok0 = (blk0 + warp + kWarps * (c / cpb)) * b + (c % cpb) * kChunkRows;  // first token

    // S = Q K^T for the chunk's 16 tokens: n-tile 0 = tokens 0-7, n-tile 1 = tokens 8-15
    float s0[4] = {0.0f, 0.0f, 0.0f, 0.0f}, s1[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
    for (int ks = 0; ks < D / 16; ++ks) {
      uint32_t kf[4];
      ldmatrix_x4(kbuf + swz_off<D>(lrow, 2 * ks + lgrp), kf);
      const uint32_t aq[4] = {qa[ks][0], 0u, qa[ks][1], 0u};
      mma_16816_bf16(s0, aq, kf[0], kf[2]);
      mma_16816_bf16(s1, aq, kf[1], kf[3]);
    }
    // online softmax of row fr over the 16 tokens (this thread: tokens 2q, 2q+1, 8+2q, 9+2q)
    const int t0 = tok0 + 2 * q;
    float sv[4] = {(t0 < seq) ? s0[0] * a.sl2 : -INFINITY, (t0 + 1 < seq) ? s0[1] * a.sl2 : -INFINITY,
                   (t0 + 8 < seq) ? s1[0] * a.sl2 : -INFINITY, (t0 + 9 < seq) ? s1[1] * a.sl2 : -INFINITY};
    float cm = fmaxf(fmaxf(sv[0], sv[1]), fmaxf(sv[2], sv[3]));
    cm = fmaxf(cm, __shfl_xor_sync(0xffffffffu, cm, 1));
    cm = fmaxf(cm, __shfl_xor_sync(0xffffffffu, cm, 2));
    const float mn = fmaxf(m, cm);
    if (mn != -INFINITY) {  // uniform over the quad; false only for a fully masked chunk
      const float corr = ex2(m - mn);
      m = mn;
      l *= corr;
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        o[nt][0] *= corr;
        o[nt][1] *= corr;
      }
      float p[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        p[e] = ex2(sv[e] - mn);
        l += p[e];
      }
      // P as A fragments, split into a bf16 high part and a bf16 remainder so that P V keeps
      // about 16 bits of P (the exp-sum l uses the fp32 values)
      const uint32_t h01 = pack_bf16x2(p[0], p[1]), h23 = pack_bf16x2(p[2], p[3]);
      const uint32_t l01 = pack_bf16x2(p[0] - bf16x2_lo(h01), p[1] - bf16x2_hi(h01));
      const uint32_t l23 = pack_bf16x2(p[2] - bf16x2_lo(h23), p[3] - bf16x2_hi(h23));
      const uint32_t ph_[4] = {h01, 0u, h23, 0u}, pl_[4] = {l01, 0u, l23, 0u};
#pragma unroll
      for (int np = 0; np < NT / 2; ++np) {  // pairs of n-tiles: columns 16np .. 16np + 15
        uint32_t vf[4];
        ldmatrix_x4_trans(vbuf + swz_off<D>(lrow, 2 * np + lgrp), vf);
        mma_16816_bf16(o[2 * np], ph_, vf[0], vf[1]);
        mma_16816_bf16(o[2 * np], pl_, vf[0], vf[1]);
        mma_16816_bf16(o[2 * np + 1], ph_, vf[2], vf[3]);
        mma_16816_bf16(o[2 * np + 1], pl_, vf[2], vf[3]);
      }
    }
    __syncwarp();  // every lane is done with stage st before it is refilled
    if (c + 2 < nch) issue(c + 2, st);
  }
  // copies still in flight after a failed wait: wait for them (bounded) before the CTA ends
  if (!ok) {
    if (lane == 0)
      for (int k = c; k < min(nch, c + 2); ++k) mbar_wait_bounded(&sm_bar[warp][k & 1], (ph >> (k & 1)) & 1u, kWaitNsD);
    atomicCAS(a.err, 0, ZP_ERR_TIMEOUT);
  }
  if (bad) atomicCAS(a.err, 0, ZP_ERR_BAD_TABLE);
  l += __shfl_xor_sync(0xffffffffu, l, 1);
  l += __shfl_xor_sync(0xffffffffu, l, 2);

  if (fr < G) {
    if (q == 0) {
      sm_m[warp][fr] = m;
      sm_l[warp][fr] = l;
    }
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      sm_acc[warp][fr][8 * nt + 2 * q] = o[nt][0];
      sm_acc[warp][fr][8 * nt + 2 * q + 1] = o[nt][1];
    }
  }
  __syncthreads();
  // merge the warps: thread -> (g, dim) pairs; a request of one split writes its output here,
  // longer ones write partials for decode_combine_kernel
  const bool single = nblk <= a.bps;
  for (int idx = tid; idx < G * D; idx += kThreads) {
    const int g = idx / D, dim = idx % D;
    float M = -INFINITY;
#pragma unroll
    for (int ww = 0; ww < kWarps; ++ww) M = fmaxf(M, sm_m[ww][g]);
    float Ls = 0.0f, As = 0.0f;
    if (M != -INFINITY)
#pragma unroll
      for (int ww = 0; ww < kWarps; ++ww) {
        const float mw = sm_m[ww][g];
        if (mw == -INFINITY) continue;
        const float cw = ex2(mw - M);
        Ls += sm_l[ww][g] * cw;
        As += sm_acc[ww][g][dim] * cw;
      }
    const int qh = h * G + g;
    if (single) {
      a.out[(static_cast<int64_t>(r) * a.Hq + qh) * D + dim] = f2bf16(Ls > 0.0f ? As / Ls : 0.0f);
    } else {
      float* p = a.part + ((static_cast<int64_t>(r) * a.Hq + qh) * a.max_splits + split) * (D + 2);
      p[dim] = As;
      if (dim == 0) {
        p[D] = M;
        p[D + 1] = Ls;
      }
    }
  }
}

// Merges the split partials of one (request, query head): grid (Hq, B), D threads.
template <int D>
__global__ void __launch_bounds__(D) decode_combine_kernel(const DecodeArgs a) {
  const int qh = blockIdx.x, r = blockIdx.y, dim = threadIdx.x;
  const int seq = a.seq_lens[r];
  if (seq < 1 || seq > a.max_blocks * a.b) return;
  const int nblk = (seq + a.b - 1) / a.b;
  const int ns = (nblk + a.bps - 1) / a.bps;
  if (ns == 1) return;  // written by the decode kernel itself
  const float* p = a.part + (static_cast<int64_t>(r) * a.Hq + qh) * a.max_splits * (D + 2);
  float M = -INFINITY;
  for (int s = 0; s < ns; ++s) M = fmaxf(M, p[s * (D + 2) + D]);
  float Ls = 0.0f, As = 0.0f;
  if (M != -INFINITY)
    for (int s = 0; s < ns; ++s) {
      const float ms = p[s * (D + 2) + D];
      if (ms == -INFINITY) continue;
      const float c = ex2(ms - M);
      Ls += p[s * (D + 2) + D + 1] * c;
      As += p[s * (D + 2) + dim] * c;
    }
  a.out[(static_cast<int64_t>(r) * a.Hq + qh) * D + dim] = f2bf16(Ls > 0.0f ? As / Ls : 0.0f);
}

template <int D, int G>
cudaError_t launch_decode(const CUtensorMap& tm, const DecodeArgs& a, cudaStream_t st) {
  constexpr int kv_bytes = kWarps * 2 * 2 * kChunkRows * D * 2 + 1024;  // + alignment slack
  static PerDeviceInit attrs;
  const cudaError_t attr = attrs.run(
      [] { return cudaFuncSetAttribute(decode_kernel<D, G>, cudaFuncAttributeMaxDynamicSharedMemorySize, kv_bytes); });
  if (attr != cudaSuccess) return attr;
  decode_kernel<D, G><<<dim3(a.max_splits, a.Hkv, a.B), kThreads, kv_bytes, st>>>(tm, a);
  if (a.max_splits > 1) decode_combine_kernel<D><<<dim3(a.Hq, a.B), D, 0, st>>>(a);
  return cudaGetLastError();
}

template <int D>
cudaError_t dispatch_g(const CUtensorMap& tm, const DecodeArgs& a, cudaStream_t st) {
  switch (a.Gq) {
    case 1: return launch_decode<D, 1>(tm, a, st);
    case 2: return launch_decode<D, 2>(tm, a, st);
    case 4: return launch_decode<D, 4>(tm, a, st);
    case 7: return launch_decode<D, 7>(tm, a, st);
    case 8: return launch_decode<D, 8>(tm, a, st);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

int decode_max_splits(int max_blocks) { return (max_blocks + kMinBlocksPerSplit - 1) / kMinBlocksPerSplit; }

// Blocks per split of a launch: the longest split that still gives about two waves of CTAs
// (three CTAs per SM).  Fewer splits mean fewer partials to merge; more splits keep every SM
// busy on small batches.
int decode_blocks_per_split(int B, int Hkv, int max_blocks) {
  for (int bps = kMaxBlocksPerSplit; bps > kMinBlocksPerSplit; bps >>= 1)
    if (static_cast<int64_t>(B) * Hkv * ((max_blocks + bps - 1) / bps) >= 6LL * num_sms()) return bps;
  return kMinBlocksPerSplit;
}

zp_status decode_validate(const zp_kv_pool* pool, int32_t layer, const uint16_t* q, const int32_t* block_tables,
                          const int32_t* seq_lens, int32_t B, int32_t max_blocks, const uint16_t* out,
                          const zp_params* p) {
  if (!pool || !q || !block_tables || !seq_lens || !out || !p || !pool->base) return ZP_ERR_INVALID_ARG;
  if (B < 0 || max_blocks < 1 || layer < 0 || layer >= p->num_layers || pool->num_blocks <= 0)
    return ZP_ERR_INVALID_ARG;
  if (p->num_kv_heads <= 0 || p->num_q_heads % p->num_kv_heads != 0) return ZP_ERR_INVALID_ARG;
  if (p->head_dim != 64 && p->head_dim != 128) return ZP_ERR_UNSUPPORTED;
  if (p->block_size != 16 && p->block_size != 32) return ZP_ERR_UNSUPPORTED;
  const int G = p->num_q_heads / p->num_kv_heads;
  if (G != 1 && G != 2 && G != 4 && G != 7 && G != 8) return ZP_ERR_UNSUPPORTED;
  if (B > 65535 || p->num_kv_heads > 65535) return ZP_ERR_UNSUPPORTED;
  if (!aligned(pool->base, 16) || !aligned(q, 16)) return ZP_ERR_INVALID_ARG;
  return ZP_OK;
}

// Launches the decode kernels with partials in `part` and the error word at `err`.
zp_status decode_launch(const zp_kv_pool* pool, int32_t layer, const uint16_t* q, const int32_t* block_tables,
                        const int32_t* seq_lens, int32_t B, int32_t max_blocks, uint16_t* out, const zp_params* p,
                        float* part, int32_t* err, cudaStream_t st, uint64_t stall_ns = 0) {
  DecodeArgs a{};
  a.pool = static_cast<const uint8_t*>(pool->base);
  a.num_blocks = pool->num_blocks;
  a.q = q;
  a.tables = block_tables;
  a.seq_lens = seq_lens;
  a.out = out;
  a.part = part;
  a.err = err;
  a.B = B;
  a.layer = layer;
  a.Hq = p->num_q_heads;
  a.Hkv = p->num_kv_heads;
  a.d = p->head_dim;
  a.b = p->block_size;
  a.Gq = p->num_q_heads / p->num_kv_heads;
  a.max_blocks = max_blocks;
  a.bps = decode_blocks_per_split(B, a.Hkv, max_blocks);
  a.max_splits = (max_blocks + a.bps - 1) / a.bps;
  a.sl2 = p->scale * 1.4426950408889634f;
  a.stall_ns = stall_ns;
  if (B == 0) return ZP_OK;
  // the pool as {d, 2*Hkv*b rows per (layer, block), layers*num_blocks}; box = 16 rows of one
  // (K or V, head) tile, 64 columns, 128-byte swizzle
  CUtensorMap tm;
  if (!encode_tmap_3d_bf16(&tm, pool->base, a.d, static_cast<uint64_t>(2) * a.Hkv * a.b,
                           static_cast<uint64_t>(p->num_layers) * pool->num_blocks, static_cast<uint64_t>(a.d) * 2,
                           static_cast<uint64_t>(2) * a.Hkv * a.b * a.d * 2, 64, kChunkRows, 1))
    return ZP_ERR_CUDA;
  const cudaError_t e = (a.d == 128) ? dispatch_g<128>(tm, a, st) : dispatch_g<64>(tm, a, st);
  return e == cudaSuccess ? ZP_OK : ZP_ERR_CUDA;
}

}  // namespace zp

using namespace zp;

extern "C" int32_t zp_paged_decode_kernel_launches(const zp_params* p, int32_t B, int32_t max_blocks) {
  if (!p || B < 1 || max_blocks < 1 || p->num_kv_heads < 1) return 0;
  const int bps = decode_blocks_per_split(B, p->num_kv_heads, max_blocks);
  return (max_blocks + bps - 1) / bps > 1 ? 2 : 1;
}

extern "C" size_t zp_paged_decode_workspace_size(const zp_params* p, int32_t B, int32_t max_blocks) {
  if (!p || B < 0 || max_blocks < 1) return 0;
  const size_t splits = static_cast<size_t>(decode_max_splits(max_blocks));
  return 256 + static_cast<size_t>(B) * p->num_q_heads * splits * (p->head_dim + 2) * sizeof(float);
}

extern "C" zp_status zp_paged_decode_attn(const zp_kv_pool* pool, int32_t layer, const uint16_t* q,
                                          const int32_t* block_tables, const int32_t* seq_lens, int32_t B,
                                          int32_t max_blocks, uint16_t* out, const zp_params* p, void* workspace,
                                          size_t workspace_bytes, zp_stream stream) {
  zp::NvtxRange nvtx_range("zp_paged_decode_attn");
  zp_status s = decode_validate(pool, layer, q, block_tables, seq_lens, B, max_blocks, out, p);
  if (s != ZP_OK) return s;
  if (!workspace || !aligned(workspace, 256) || workspace_bytes < zp_paged_decode_workspace_size(p, B, max_blocks))
    return ZP_ERR_INVALID_ARG;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (cudaMemsetAsync(workspace, 0, 4, st) != cudaSuccess) return ZP_ERR_CUDA;
  float* part = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + 256);
  return decode_launch(pool, layer, q, block_tables, seq_lens, B, max_blocks, out, p, part,
                       static_cast<int32_t*>(workspace), st);
}

extern "C" zp_status zp_test_decode_stalled(const zp_kv_pool* pool, int32_t layer, const uint16_t* q,
                                            const int32_t* block_tables, const int32_t* seq_lens, int32_t B,
                                            int32_t max_blocks, uint16_t* out, const zp_params* p,
                                            void* workspace, size_t workspace_bytes, int64_t stall_limit_ns,
                                            zp_stream stream) {
  zp::NvtxRange nvtx_range("zp_test_decode_stalled");
  if (stall_limit_ns < 1 || stall_limit_ns > 1000000000LL) return ZP_ERR_INVALID_ARG;
  zp_status s = decode_validate(pool, layer, q, block_tables, seq_lens, B, max_blocks, out, p);
  if (s != ZP_OK) return s;
  if (!workspace || !aligned(workspace, 256) || workspace_bytes < zp_paged_decode_workspace_size(p, B, max_blocks))
    return ZP_ERR_INVALID_ARG;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (cudaMemsetAsync(workspace, 0, 4, st) != cudaSuccess) return ZP_ERR_CUDA;
  float* part = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + 256);
  return decode_launch(pool, layer, q, block_tables, seq_lens, B, max_blocks, out, p, part,
                       static_cast<int32_t*>(workspace), st, static_cast<uint64_t>(stall_limit_ns));
}

// ------------------------------------------------------------------ no-allocation variant ----
//
// Scratch for zp_paged_decode_attn_static: the split-KV partials (and a spare error word) of
// decode attention live in this fixed device array instead of a caller workspace.  Every GPU
// that loads the library holds these 16 MiB until the process exits.  In host code the name
// is only a host-side stand-in; the device address is obtained with cudaGetSymbolAddress,
// once per device, while that device is current.
namespace {
constexpr size_t kStaticScratchBytes = size_t(16) << 20;
constexpr size_t kStaticErrBytes = 256;  // spare error word when the caller passes no status
constexpr int kMaxDevicesStatic = 64;
std::mutex g_static_mu;
void* g_static_addr[kMaxDevicesStatic] = {};
}  // namespace

static __device__ __align__(256) unsigned char g_decode_static_scratch[kStaticScratchBytes];

extern "C" zp_status zp_paged_decode_attn_static(const zp_kv_pool* pool, int32_t layer, const uint16_t* q,
                                                 const int32_t* block_tables, const int32_t* seq_lens,
                                                 int32_t B, int32_t max_blocks, uint16_t* out,
                                                 const zp_params* p, int32_t* dev_status, zp_stream stream) {
  zp::NvtxRange nvtx_range("zp_paged_decode_attn_static");
  zp_status s = decode_validate(pool, layer, q, block_tables, seq_lens, B, max_blocks, out, p);
  if (s != ZP_OK) return s;
  const size_t need = zp_paged_decode_workspace_size(p, B, max_blocks) - 256;  // partials only
  if (need > kStaticScratchBytes - kStaticErrBytes) return ZP_ERR_TOO_LARGE;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return ZP_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevicesStatic) return ZP_ERR_UNSUPPORTED;
  void* base = nullptr;
  {
    std::lock_guard<std::mutex> lock(g_static_mu);
    if (!g_static_addr[dev]) {
      void* addr = nullptr;
      if (cudaGetSymbolAddress(&addr, g_decode_static_scratch) != cudaSuccess || !addr) return ZP_ERR_CUDA;
      g_static_addr[dev] = addr;
    }
    base = g_static_addr[dev];
  }
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  int32_t* err = dev_status ? dev_status : static_cast<int32_t*>(base);
  if (cudaMemsetAsync(err, 0, sizeof(int32_t), st) != cudaSuccess) return ZP_ERR_CUDA;
  float* part = reinterpret_cast<float*>(static_cast<uint8_t*>(base) + kStaticErrBytes);
  return decode_launch(pool, layer, q, block_tables, seq_lens, B, max_blocks, out, p, part, err, st);
}
