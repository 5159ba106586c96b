// zp_decode.cu — paged decode attention over the (compacted) KV cache, sm_103a.
//
// The consumer of the compression pass: requests that are not compressing keep decoding
// while compression runs on a side stream (Zipage summaries on gist.science: zh §2.1
// asynchronous compression and decoding, zh §2.3 PagedAttention/FlashAttention integration,
// fr §2.D).  One new token per request and one layer per launch:
//   out[r][qh] = sum_t softmax_t(scale * <q[r][qh], k_t>) v_t,  t < seq_lens[r],
// with k_t, v_t of kv head qh / G_q read through block_tables[r].
//
// Split-KV flash decoding.  Grid (split, kv head, request); each CTA of 4 warps walks its
// split's blocks (warp w takes blocks w, w+4, ...).  A token's 256-byte K row is spread over
// d/8 lanes (16 bytes each), so one warp-wide 16-byte load covers 32*16 bytes of K; the G_q
// query heads of the kv head share every K/V byte loaded.  Each lane group keeps an online
// softmax (log2 domain) per query head; groups, then warps, are merged at the end.  With
// more than one split the (max, sum, acc) partials go to the workspace and a second kernel
// merges the splits.
#include "zp_internal.h"
#include "zp_ptx.cuh"

#include <mutex>

namespace zp {
namespace {

constexpr int kWarps = 4;
constexpr int kThreads = kWarps * 32;
constexpr int kBlocksPerSplit = 16;  // KV blocks per CTA

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
  float sl2;  // scale * log2(e)
};

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ float bf16_lo(uint32_t u) { return __uint_as_float(u << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t u) { return __uint_as_float(u & 0xFFFF0000u); }

__device__ __forceinline__ uint16_t f2bf16(float f) {
  // round to nearest even; NaN stays NaN
  uint32_t u = __float_as_uint(f);
  if ((u & 0x7FFFFFFFu) > 0x7F800000u) return static_cast<uint16_t>((u >> 16) | 0x40u);
  u += 0x7FFFu + ((u >> 16) & 1u);
  return static_cast<uint16_t>(u >> 16);
}

template <int D, int G>
__global__ void __launch_bounds__(kThreads) decode_kernel(const DecodeArgs a) {
  constexpr int LPT = D / 8;        // lanes per token
  constexpr int TPS = 32 / LPT;     // tokens per warp step
  constexpr int kStepsPerChunk = (G <= 4) ? 8 : 4;  // 16-byte lane loads in flight per chunk
  __shared__ float sm_m[kWarps][G], sm_l[kWarps][G];
  __shared__ float sm_acc[kWarps][G][D];
  __shared__ int sm_bad;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int split = blockIdx.x, h = blockIdx.y, r = blockIdx.z;
  const int sub = lane % LPT;       // which 16-byte chunk of the row
  const int grp = lane / LPT;       // which token of the step
  const int seq = a.seq_lens[r];
  const int b = a.b;
  const int nblk = (seq + b - 1) / b;
  const int blk0 = split * kBlocksPerSplit;
  const int blk1 = min(nblk, blk0 + kBlocksPerSplit);

  if (tid == 0) sm_bad = (seq < 1 || seq > a.max_blocks * b) ? 1 : 0;
  __syncthreads();
  if (sm_bad) {
    if (tid == 0 && split == 0 && h == 0) atomicCAS(a.err, 0, ZP_ERR_BAD_TABLE);
    return;
  }
  if (blk0 >= nblk) return;  // this split has no work (uniform over the CTA)

  // query chunk of this lane, pre-scaled into the log2 domain
  float qf[G][8];
#pragma unroll
  for (int g = 0; g < G; ++g) {
    const uint4 raw = *reinterpret_cast<const uint4*>(a.q + (static_cast<int64_t>(r) * a.Hq + h * G + g) * D + sub * 8);
    const uint32_t w4[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      qf[g][2 * i] = bf16_lo(w4[i]) * a.sl2;
      qf[g][2 * i + 1] = bf16_hi(w4[i]) * a.sl2;
    }
  }
  float m[G], l[G], acc[G][8];
#pragma unroll
  for (int g = 0; g < G; ++g) {
    m[g] = -INFINITY;
    l[g] = 0.0f;
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[g][i] = 0.0f;
  }

  const int32_t* table = a.tables + static_cast<int64_t>(r) * a.max_blocks;
  const int64_t tile_elems = static_cast<int64_t>(b) * D;
  bool bad = false;
  for (int blk = blk0 + warp; blk < blk1; blk += kWarps) {
    const int phys = table[blk];
    if (phys < 0 || phys >= a.num_blocks) {
      bad = true;
      continue;
    }
    const uint16_t* kbase =
        reinterpret_cast<const uint16_t*>(a.pool) +
        ((static_cast<int64_t>(a.layer) * a.num_blocks + phys) * 2 * a.Hkv + h) * tile_elems;
    const uint16_t* vbase = kbase + static_cast<int64_t>(a.Hkv) * tile_elems;
    for (int t0 = 0; t0 < b; t0 += kStepsPerChunk * TPS) {
      uint4 kr[kStepsPerChunk];
#pragma unroll
      for (int s = 0; s < kStepsPerChunk; ++s) {
        const int t = t0 + s * TPS + grp;
        kr[s] = (t < b) ? *reinterpret_cast<const uint4*>(kbase + static_cast<int64_t>(t) * D + sub * 8)
                        : make_uint4(0, 0, 0, 0);
      }
      float sc[kStepsPerChunk][G];
#pragma unroll
      for (int s = 0; s < kStepsPerChunk; ++s) {
        const uint32_t w4[4] = {kr[s].x, kr[s].y, kr[s].z, kr[s].w};
        float kf[8];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          kf[2 * i] = bf16_lo(w4[i]);
          kf[2 * i + 1] = bf16_hi(w4[i]);
        }
#pragma unroll
        for (int g = 0; g < G; ++g) {
          float p = 0.0f;
#pragma unroll
          for (int i = 0; i < 8; ++i) p = fmaf(qf[g][i], kf[i], p);
#pragma unroll
          for (int off = LPT / 2; off >= 1; off >>= 1) p += __shfl_xor_sync(0xffffffffu, p, off);
          const int tok = blk * b + t0 + s * TPS + grp;
          sc[s][g] = (t0 + s * TPS + grp < b && tok < seq) ? p : -INFINITY;
        }
      }
      uint4 vr[kStepsPerChunk];
#pragma unroll
      for (int s = 0; s < kStepsPerChunk; ++s) {
        const int t = t0 + s * TPS + grp;
        vr[s] = (t < b) ? *reinterpret_cast<const uint4*>(vbase + static_cast<int64_t>(t) * D + sub * 8)
                        : make_uint4(0, 0, 0, 0);
      }
#pragma unroll
      for (int g = 0; g < G; ++g) {
        float cm = m[g];
#pragma unroll
        for (int s = 0; s < kStepsPerChunk; ++s) cm = fmaxf(cm, sc[s][g]);
        if (cm == -INFINITY) continue;
        const float corr = ex2(m[g] - cm);
        m[g] = cm;
        l[g] *= corr;
#pragma unroll
        for (int i = 0; i < 8; ++i) acc[g][i] *= corr;
#pragma unroll
        for (int s = 0; s < kStepsPerChunk; ++s) {
          const float p = ex2(sc[s][g] - cm);
          l[g] += p;
          const uint32_t w4[4] = {vr[s].x, vr[s].y, vr[s].z, vr[s].w};
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            acc[g][2 * i] = fmaf(p, bf16_lo(w4[i]), acc[g][2 * i]);
            acc[g][2 * i + 1] = fmaf(p, bf16_hi(w4[i]), acc[g][2 * i + 1]);
          }
        }
      }
    }
  }
  if (bad) atomicCAS(a.err, 0, ZP_ERR_BAD_TABLE);

  // merge the TPS token groups of the warp (same dims, different tokens)
#pragma unroll
  for (int off = 16; off >= LPT; off >>= 1) {
#pragma unroll
    for (int g = 0; g < G; ++g) {
      const float mo = __shfl_xor_sync(0xffffffffu, m[g], off);
      const float lo = __shfl_xor_sync(0xffffffffu, l[g], off);
      const float mn = fmaxf(m[g], mo);
      const float c0 = (m[g] == -INFINITY) ? 0.0f : ex2(m[g] - mn);
      const float c1 = (mo == -INFINITY) ? 0.0f : ex2(mo - mn);
      l[g] = l[g] * c0 + lo * c1;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const float ao = __shfl_xor_sync(0xffffffffu, acc[g][i], off);
        acc[g][i] = acc[g][i] * c0 + ao * c1;
      }
      m[g] = mn;
    }
  }
  if (lane < LPT) {
#pragma unroll
    for (int g = 0; g < G; ++g) {
      if (lane == 0) {
        sm_m[warp][g] = m[g];
        sm_l[warp][g] = l[g];
      }
#pragma unroll
      for (int i = 0; i < 8; ++i) sm_acc[warp][g][sub * 8 + i] = acc[g][i];
    }
  }
  __syncthreads();
  // merge the warps: thread -> (g, dim) pairs
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
    if (a.max_splits == 1) {
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
  const int ns = (nblk + kBlocksPerSplit - 1) / kBlocksPerSplit;
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
cudaError_t launch_decode(const DecodeArgs& a, cudaStream_t st) {
  decode_kernel<D, G><<<dim3(a.max_splits, a.Hkv, a.B), kThreads, 0, st>>>(a);
  if (a.max_splits > 1) decode_combine_kernel<D><<<dim3(a.Hq, a.B), D, 0, st>>>(a);
  return cudaGetLastError();
}

template <int D>
cudaError_t dispatch_g(const DecodeArgs& a, cudaStream_t st) {
  switch (a.Gq) {
    case 1: return launch_decode<D, 1>(a, st);
    case 2: return launch_decode<D, 2>(a, st);
    case 4: return launch_decode<D, 4>(a, st);
    case 7: return launch_decode<D, 7>(a, st);
    case 8: return launch_decode<D, 8>(a, st);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

int decode_max_splits(int max_blocks) { return (max_blocks + kBlocksPerSplit - 1) / kBlocksPerSplit; }

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
                        float* part, int32_t* err, cudaStream_t st) {
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
  a.max_splits = decode_max_splits(max_blocks);
  a.sl2 = p->scale * 1.4426950408889634f;
  if (B == 0) return ZP_OK;
  const cudaError_t e = (a.d == 128) ? dispatch_g<128>(a, st) : dispatch_g<64>(a, st);
  return e == cudaSuccess ? ZP_OK : ZP_ERR_CUDA;
}

}  // namespace zp

using namespace zp;

extern "C" size_t zp_paged_decode_workspace_size(const zp_params* p, int32_t B, int32_t max_blocks) {
  if (!p || B < 0 || max_blocks < 1) return 0;
  const size_t splits = static_cast<size_t>(decode_max_splits(max_blocks));
  return 256 + static_cast<size_t>(B) * p->num_q_heads * splits * (p->head_dim + 2) * sizeof(float);
}

extern "C" zp_status zp_paged_decode_attn(const zp_kv_pool* pool, int32_t layer, const uint16_t* q,
                                          const int32_t* block_tables, const int32_t* seq_lens, int32_t B,
                                          int32_t max_blocks, uint16_t* out, const zp_params* p, void* workspace,
                                          size_t workspace_bytes, zp_stream stream) {
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
