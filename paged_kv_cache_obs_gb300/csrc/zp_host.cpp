// zp_host.cpp — host side of the library: tensor-map encoding, the device error word, and the
// refcounted block allocator with deferred release and the compression planner.
//
// The allocator is the PagedAttention block manager with prefix sharing that Compressed
// PagedAttention builds on (Zipage summaries on gist.science: zh §2.2 prefix-cache
// compatibility, de §2 "Prefix Caching für komprimierte Daten", fr §2.C): a block shared by
// several requests (refcount > 1) must not be rewritten, so compression redirects the
// survivors of a shared leading block into a freshly allocated target block.  The last block
// of a compressed request is released (zh §2.1) once the compression kernel that still reads
// it has finished, which is what the event-deferred decref provides.
#include <algorithm>
#include <cstring>
#include <mutex>
#include <new>
#include <set>
#include <vector>

#include "zp_internal.h"

namespace zp {

namespace {
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn get_encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    cudaDriverEntryPointQueryResult q;
    void* p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}
}  // namespace

bool encode_tmap_3d_bf16(CUtensorMap* map, const void* base, uint64_t d0, uint64_t d1, uint64_t d2,
                         uint64_t stride1_bytes, uint64_t stride2_bytes, uint32_t box0, uint32_t box1,
                         uint32_t box2) {
  EncodeTiledFn fn = get_encode_fn();
  if (!fn) return false;
  cuuint64_t dims[3] = {d0, d1, d2};
  cuuint64_t strides[2] = {stride1_bytes, stride2_bytes};
  cuuint32_t box[3] = {box0, box1, box2};
  cuuint32_t elem[3] = {1, 1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, elem,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int num_sms() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  return n;
}

}  // namespace zp

// ------------------------------------------------------------------ allocator -------------

struct PendingDecref {
  cudaEvent_t event;
  std::vector<int32_t> ids;
};

struct zp_alloc {
  std::vector<int32_t> refcount;
  std::set<int32_t> free_ids;  // ordered: lowest id first
  std::vector<PendingDecref> pending;
  // host-side fault injection for tests: the n-th allocation from now fails (0 = never)
  int64_t fail_after = 0;
};

namespace {

bool valid_id(const zp_alloc* a, int32_t id) {
  return id >= 0 && static_cast<size_t>(id) < a->refcount.size();
}

zp_status apply_decref(zp_alloc* a, const int32_t* ids, int32_t n) {
  // all-or-nothing: check first (an id may appear several times)
  std::vector<std::pair<int32_t, int32_t>> counts;
  counts.reserve(n);
  for (int32_t i = 0; i < n; ++i) {
    if (!valid_id(a, ids[i])) return ZP_ERR_INVALID_ARG;
    counts.emplace_back(ids[i], 1);
  }
  std::sort(counts.begin(), counts.end());
  for (size_t i = 0; i < counts.size();) {
    size_t j = i;
    int32_t c = 0;
    while (j < counts.size() && counts[j].first == counts[i].first) c += counts[j++].second;
    if (a->refcount[counts[i].first] < c) return ZP_ERR_INVALID_ARG;
    i = j;
  }
  for (int32_t i = 0; i < n; ++i)
    if (--a->refcount[ids[i]] == 0) a->free_ids.insert(ids[i]);
  return ZP_OK;
}

// Applies the pending decrefs whose events have completed (in order of submission).
zp_status poll_pending(zp_alloc* a, bool wait) {
  size_t done = 0;
  for (; done < a->pending.size(); ++done) {
    PendingDecref& p = a->pending[done];
    if (p.event) {
      cudaError_t e = wait ? cudaEventSynchronize(p.event) : cudaEventQuery(p.event);
      if (e == cudaErrorNotReady) break;
      if (e != cudaSuccess) return ZP_ERR_CUDA;
      cudaEventDestroy(p.event);
      p.event = nullptr;
    }
    zp_status s = apply_decref(a, p.ids.data(), static_cast<int32_t>(p.ids.size()));
    if (s != ZP_OK) return s;
  }
  a->pending.erase(a->pending.begin(), a->pending.begin() + done);
  return ZP_OK;
}

}  // namespace

extern "C" {

int32_t zp_version(void) { return 1; }

zp_status zp_alloc_create(int64_t num_blocks, zp_alloc** out) {
  if (!out || num_blocks <= 0 || num_blocks > INT32_MAX) return ZP_ERR_INVALID_ARG;
  zp_alloc* a = new (std::nothrow) zp_alloc();
  if (!a) return ZP_ERR_NO_BLOCKS;
  a->refcount.assign(static_cast<size_t>(num_blocks), 0);
  for (int64_t i = 0; i < num_blocks; ++i) a->free_ids.insert(static_cast<int32_t>(i));
  *out = a;
  return ZP_OK;
}

void zp_alloc_destroy(zp_alloc* a) {
  if (!a) return;
  for (auto& p : a->pending)
    if (p.event) {
      cudaEventSynchronize(p.event);
      cudaEventDestroy(p.event);
    }
  delete a;
}

zp_status zp_alloc_blocks(zp_alloc* a, int32_t n, int32_t* ids) {
  if (!a || n < 0 || (n > 0 && !ids)) return ZP_ERR_INVALID_ARG;
  poll_pending(a, false);
  if (static_cast<int64_t>(a->free_ids.size()) < n) return ZP_ERR_NO_BLOCKS;
  if (a->fail_after > 0 && --a->fail_after == 0) return ZP_ERR_NO_BLOCKS;
  auto it = a->free_ids.begin();
  for (int32_t i = 0; i < n; ++i) {
    ids[i] = *it;
    a->refcount[*it] = 1;
    it = a->free_ids.erase(it);
  }
  return ZP_OK;
}

zp_status zp_alloc_reserve(zp_alloc* a, const int32_t* ids, int32_t n) {
  if (!a || n < 0 || (n > 0 && !ids)) return ZP_ERR_INVALID_ARG;
  std::vector<int32_t> v(ids, ids + n);
  std::sort(v.begin(), v.end());
  for (int32_t i = 0; i < n; ++i) {
    if (!valid_id(a, v[i]) || a->refcount[v[i]] != 0) return ZP_ERR_INVALID_ARG;
    if (i > 0 && v[i] == v[i - 1]) return ZP_ERR_INVALID_ARG;
  }
  for (int32_t id : v) {
    a->refcount[id] = 1;
    a->free_ids.erase(id);
  }
  return ZP_OK;
}

zp_status zp_incref(zp_alloc* a, const int32_t* ids, int32_t n) {
  if (!a || n < 0 || (n > 0 && !ids)) return ZP_ERR_INVALID_ARG;
  for (int32_t i = 0; i < n; ++i)
    if (!valid_id(a, ids[i]) || a->refcount[ids[i]] <= 0) return ZP_ERR_INVALID_ARG;
  for (int32_t i = 0; i < n; ++i) ++a->refcount[ids[i]];
  return ZP_OK;
}

zp_status zp_decref(zp_alloc* a, const int32_t* ids, int32_t n) {
  if (!a || n < 0 || (n > 0 && !ids)) return ZP_ERR_INVALID_ARG;
  return apply_decref(a, ids, n);
}

zp_status zp_decref_after(zp_alloc* a, const int32_t* ids, int32_t n, zp_stream stream) {
  if (!a || n < 0 || (n > 0 && !ids)) return ZP_ERR_INVALID_ARG;
  for (int32_t i = 0; i < n; ++i)
    if (!valid_id(a, ids[i])) return ZP_ERR_INVALID_ARG;
  PendingDecref p;
  p.event = nullptr;
  p.ids.assign(ids, ids + n);
  if (stream) {
    if (cudaEventCreateWithFlags(&p.event, cudaEventDisableTiming) != cudaSuccess) return ZP_ERR_CUDA;
    if (cudaEventRecord(p.event, reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess) {
      cudaEventDestroy(p.event);
      return ZP_ERR_CUDA;
    }
  }
  a->pending.push_back(std::move(p));
  return poll_pending(a, false);
}

zp_status zp_alloc_poll(zp_alloc* a) {
  if (!a) return ZP_ERR_INVALID_ARG;
  return poll_pending(a, false);
}

zp_status zp_alloc_drain(zp_alloc* a) {
  if (!a) return ZP_ERR_INVALID_ARG;
  return poll_pending(a, true);
}

int32_t zp_refcount(const zp_alloc* a, int32_t id) {
  if (!a || !valid_id(a, id)) return -1;
  return a->refcount[id];
}

int64_t zp_num_free(const zp_alloc* a) { return a ? static_cast<int64_t>(a->free_ids.size()) : -1; }

int64_t zp_num_pending(const zp_alloc* a) {
  if (!a) return -1;
  int64_t n = 0;
  for (const auto& p : a->pending) n += static_cast<int64_t>(p.ids.size());
  return n;
}

// Test hook: the n-th allocation call from now fails with ZP_ERR_NO_BLOCKS (0 disables).
zp_status zp_alloc_inject_failure(zp_alloc* a, int64_t nth_call) {
  if (!a || nth_call < 0) return ZP_ERR_INVALID_ARG;
  a->fail_after = nth_call;
  return ZP_OK;
}

namespace {
// Plan with a budget per request (host_n_max) or one budget for all (n_max_all).
zp_status plan_impl(zp_alloc* a, const int32_t* host_tables, int32_t R, int32_t max_blocks, const int32_t* host_n_max,
                    int32_t n_max_all, int32_t* host_dst_tables) {
  if (!a || R < 0 || (R > 0 && (!host_tables || !host_dst_tables))) return ZP_ERR_INVALID_ARG;
  auto nmax_of = [&](int32_t r) { return host_n_max ? host_n_max[r] : n_max_all; };
  for (int32_t r = 0; r < R; ++r)
    if (nmax_of(r) < 2 || nmax_of(r) > max_blocks) return ZP_ERR_INVALID_ARG;
  poll_pending(a, false);
  int64_t need = 0;
  for (int32_t r = 0; r < R; ++r)
    for (int32_t i = 0; i < nmax_of(r); ++i) {
      const int32_t id = host_tables[static_cast<int64_t>(r) * max_blocks + i];
      if (!valid_id(a, id) || a->refcount[id] <= 0) return ZP_ERR_INVALID_ARG;
      if (i < nmax_of(r) - 1 && a->refcount[id] > 1) ++need;
    }
  std::vector<int32_t> fresh(static_cast<size_t>(need));
  if (need > 0) {
    zp_status s = zp_alloc_blocks(a, static_cast<int32_t>(need), fresh.data());
    if (s != ZP_OK) return s;
  }
  size_t next = 0;
  for (int32_t r = 0; r < R; ++r)
    for (int32_t i = 0; i < max_blocks; ++i) {
      const int64_t o = static_cast<int64_t>(r) * max_blocks + i;
      const int32_t id = host_tables[o];
      if (i >= nmax_of(r) - 1) {
        host_dst_tables[o] = id;
        continue;
      }
      host_dst_tables[o] = (a->refcount[id] > 1) ? fresh[next++] : id;
    }
  return ZP_OK;
}

zp_status commit_impl(zp_alloc* a, const int32_t* old_tables, const int32_t* new_tables, int32_t R, int32_t max_blocks,
                      const int32_t* host_n_max, int32_t n_max_all, int32_t block_size, const int32_t* host_seq_len,
                      zp_stream stream) {
  if (!a || R < 0 || (R > 0 && (!old_tables || !new_tables))) return ZP_ERR_INVALID_ARG;
  if (host_seq_len && block_size <= 0) return ZP_ERR_INVALID_ARG;
  std::vector<int32_t> release;
  for (int32_t r = 0; r < R; ++r) {
    const int32_t n_max = host_n_max ? host_n_max[r] : n_max_all;
    if (n_max < 2 || n_max > max_blocks) return ZP_ERR_INVALID_ARG;
    const int32_t* o = old_tables + static_cast<int64_t>(r) * max_blocks;
    const int32_t* n = new_tables + static_cast<int64_t>(r) * max_blocks;
    for (int32_t i = 0; i < n_max - 1; ++i)
      if (o[i] != n[i]) release.push_back(o[i]);
    // every block past the first n_max - 1: one at the decode trigger, more after a prefill
    const int32_t nblk = host_seq_len ? (host_seq_len[r] + block_size - 1) / block_size : n_max;
    if (nblk < n_max || nblk > max_blocks) return ZP_ERR_INVALID_ARG;
    for (int32_t i = n_max - 1; i < nblk; ++i) release.push_back(o[i]);
  }
  return zp_decref_after(a, release.data(), static_cast<int32_t>(release.size()), stream);
}
}  // namespace

zp_status zp_plan_compress(zp_alloc* a, const int32_t* host_tables, int32_t R, int32_t max_blocks, int32_t n_max,
                           int32_t* host_dst_tables) {
  zp::NvtxRange nvtx_range("zp_plan_compress");
  if (n_max < 2 || max_blocks < n_max) return ZP_ERR_INVALID_ARG;
  return plan_impl(a, host_tables, R, max_blocks, nullptr, n_max, host_dst_tables);
}

zp_status zp_plan_compress_budgets(zp_alloc* a, const int32_t* host_tables, int32_t R, int32_t max_blocks,
                                   const int32_t* host_n_max, int32_t* host_dst_tables) {
  zp::NvtxRange nvtx_range("zp_plan_compress_budgets");
  if (!host_n_max && R > 0) return ZP_ERR_INVALID_ARG;
  return plan_impl(a, host_tables, R, max_blocks, host_n_max, 0, host_dst_tables);
}

zp_status zp_commit_compress(zp_alloc* a, const int32_t* old_tables, const int32_t* new_tables, int32_t R,
                             int32_t max_blocks, int32_t n_max, int32_t block_size, const int32_t* host_seq_len,
                             zp_stream stream) {
  zp::NvtxRange nvtx_range("zp_commit_compress");
  if (n_max < 2 || max_blocks < n_max) return ZP_ERR_INVALID_ARG;
  return commit_impl(a, old_tables, new_tables, R, max_blocks, nullptr, n_max, block_size, host_seq_len, stream);
}

zp_status zp_commit_compress_budgets(zp_alloc* a, const int32_t* old_tables, const int32_t* new_tables, int32_t R,
                                     int32_t max_blocks, const int32_t* host_n_max, int32_t n_max, int32_t block_size,
                                     const int32_t* host_seq_len, zp_stream stream) {
  zp::NvtxRange nvtx_range("zp_commit_compress_budgets");
  return commit_impl(a, old_tables, new_tables, R, max_blocks, host_n_max, n_max, block_size, host_seq_len, stream);
}

zp_status zp_read_error(void* workspace, zp_stream stream, zp_status* out_status) {
  if (!workspace || !out_status) return ZP_ERR_INVALID_ARG;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  int32_t v = 0;
  if (cudaStreamSynchronize(st) != cudaSuccess) return ZP_ERR_CUDA;
  if (cudaMemcpy(&v, workspace, sizeof(v), cudaMemcpyDeviceToHost) != cudaSuccess) return ZP_ERR_CUDA;
  if (cudaMemset(workspace, 0, sizeof(v)) != cudaSuccess) return ZP_ERR_CUDA;
  *out_status = v;
  return ZP_OK;
}

}  // extern "C"
