// zp_sched.cpp — hybrid scheduler of Compressed PagedAttention (host only).
//
// The scheduling policy the pages describe around the compression pass (Zipage summaries on
// gist.science: zh §2.2 "混合调度策略", de §2 "Hybrid Scheduling", es §2 "Scheduling Híbrido",
// fr §2.B "Stratégies de Planification Hybride"):
//   - only the first M running requests (in admission order) hold a query slot, the buffer of
//     window queries a compression needs;
//   - requests that hold fewer than N_max blocks, or whose last block is not yet full, decode
//     without a slot, so the number of running requests may exceed M;
//   - a request at N_max blocks with a full last block compresses (asynchronously, rejoining
//     the next step) if it holds a slot, and otherwise waits for one;
//   - when a new block cannot be allocated, requests without a slot are preempted first (most
//     recently admitted first; they return to the queue and recompute); when none is left the
//     scheduler falls back to restricted mode, where only slot holders run and nothing new is
//     admitted.
// The scheduler owns the request state and drives the block allocator (zp_alloc) and the
// compression planner / commit of zipage.h; it does no GPU work itself.  One zp_sched_step()
// plans one engine step; the caller runs the step (decode for the planned requests,
// zp_compress for the compressing ones) and the next zp_sched_step() applies its results.
#include <algorithm>
#include <deque>
#include <new>
#include <vector>

#include "zp_internal.h"

namespace {

enum ReqState : int32_t { kWaiting = 0, kRunning = 1, kFinished = 2 };

struct Request {
  int32_t id;
  int32_t prompt_len;
  int32_t gen_len;
  int32_t generated = 0;
  int32_t seq_len = 0;          // cached tokens
  std::vector<int32_t> table;   // physical blocks
  int32_t state = kWaiting;
  int64_t admit_order = -1;     // admission counter (slots go to the earliest running)
  bool has_slot = false;
  int32_t preemptions = 0;
};

}  // namespace

struct zp_sched {
  zp_alloc* alloc;
  zp_sched_config cfg;
  std::vector<Request> reqs;
  std::deque<int32_t> waiting;        // request ids, FIFO (preempted requests go to the front)
  std::vector<int32_t> running;       // in admission order
  int64_t admit_counter = 0;
  bool restricted = false;
  // the plan of the last step (owned here, exposed through zp_sched_plan)
  std::vector<int32_t> plan_decode, plan_compress, plan_prefill, plan_preempted;
  zp_sched_stats stats{};
};

namespace {

int32_t blocks_for(const zp_sched* s, int32_t tokens) {
  return (tokens + s->cfg.block_size - 1) / s->cfg.block_size;
}

void release_all(zp_sched* s, Request& r) {
  if (!r.table.empty()) zp_decref(s->alloc, r.table.data(), static_cast<int32_t>(r.table.size()));
  r.table.clear();
}

void assign_slots(zp_sched* s) {
  // the first M running requests (admission order) hold the query slots
  int32_t given = 0;
  for (int32_t id : s->running) {
    Request& r = s->reqs[id];
    r.has_slot = given < s->cfg.num_slots;
    if (r.has_slot) ++given;
  }
}

// Preempts the most recently admitted running request without a slot (not `except`); returns
// false if there is none.
bool preempt_one(zp_sched* s, int32_t except) {
  for (auto it = s->running.rbegin(); it != s->running.rend(); ++it) {
    Request& r = s->reqs[*it];
    if (r.has_slot || r.id == except) continue;
    release_all(s, r);
    r.state = kWaiting;
    r.seq_len = 0;
    r.generated = 0;  // recomputed from the prompt when readmitted
    ++r.preemptions;
    ++s->stats.preemptions;
    s->plan_preempted.push_back(r.id);
    s->waiting.push_front(r.id);
    s->running.erase(std::next(it).base());
    return true;
  }
  return false;
}

// One fresh block for request `id`, preempting slot-less requests if the pool is exhausted.
bool grow(zp_sched* s, int32_t id) {
  int32_t blk = -1;
  while (zp_alloc_blocks(s->alloc, 1, &blk) != ZP_OK) {
    if (!preempt_one(s, id)) {
      s->restricted = true;
      return false;
    }
  }
  s->reqs[id].table.push_back(blk);
  return true;
}

}  // namespace

extern "C" {

zp_status zp_sched_create(zp_alloc* alloc, const zp_sched_config* cfg, zp_sched** out) {
  if (!alloc || !cfg || !out || cfg->n_max < 2 || cfg->block_size <= 0 || cfg->num_slots < 1) return ZP_ERR_INVALID_ARG;
  zp_sched* s = new (std::nothrow) zp_sched();
  if (!s) return ZP_ERR_NO_BLOCKS;
  s->alloc = alloc;
  s->cfg = *cfg;
  *out = s;
  return ZP_OK;
}

void zp_sched_destroy(zp_sched* s) {
  if (!s) return;
  for (Request& r : s->reqs) release_all(s, r);
  delete s;
}

zp_status zp_sched_submit(zp_sched* s, int32_t prompt_len, int32_t gen_len, int32_t* req_id) {
  if (!s || prompt_len < 1 || gen_len < 1 || !req_id) return ZP_ERR_INVALID_ARG;
  Request r;
  r.id = static_cast<int32_t>(s->reqs.size());
  r.prompt_len = prompt_len;
  r.gen_len = gen_len;
  s->reqs.push_back(r);
  s->waiting.push_back(r.id);
  ++s->stats.submitted;
  *req_id = r.id;
  return ZP_OK;
}

zp_status zp_sched_step(zp_sched* s, zp_sched_plan* plan) {
  if (!s || !plan) return ZP_ERR_INVALID_ARG;
  const int32_t b = s->cfg.block_size, n_max = s->cfg.n_max, k = (n_max - 1) * b;

  // 1. apply the previous step: decoded requests gained a token, compressed requests keep k
  //    tokens in their first n_max-1 blocks (the rest is released), finished requests leave
  for (int32_t id : s->plan_compress) {
    Request& r = s->reqs[id];
    if (r.state != kRunning) continue;
    const int32_t keep = n_max - 1;
    if (static_cast<int32_t>(r.table.size()) > keep) {
      zp_decref(s->alloc, r.table.data() + keep, static_cast<int32_t>(r.table.size()) - keep);
      r.table.resize(keep);
    }
    r.seq_len = k;
    ++s->stats.compressions;
  }
  for (int32_t id : s->plan_decode) {
    Request& r = s->reqs[id];
    if (r.state != kRunning) continue;
    ++r.seq_len;
    ++r.generated;
    ++s->stats.decoded_tokens;
    if (r.generated >= r.gen_len) {
      release_all(s, r);
      r.state = kFinished;
      r.has_slot = false;
      ++s->stats.finished;
    }
  }
  s->running.erase(std::remove_if(s->running.begin(), s->running.end(),
                                  [&](int32_t id) { return s->reqs[id].state != kRunning; }),
                   s->running.end());
  s->plan_decode.clear();
  s->plan_compress.clear();
  s->plan_prefill.clear();
  s->plan_preempted.clear();
  s->restricted = false;
  assign_slots(s);

  // 2. admit waiting requests (prefill) while their prompt's blocks are free; a prompt longer
  //    than n_max*b is admitted too (prefill may exceed the cap until the first compression)
  while (!s->waiting.empty() && (s->cfg.max_running <= 0 || static_cast<int32_t>(s->running.size()) < s->cfg.max_running)) {
    Request& r = s->reqs[s->waiting.front()];
    const int32_t need = blocks_for(s, r.prompt_len);
    std::vector<int32_t> ids(static_cast<size_t>(need));
    if (zp_alloc_blocks(s->alloc, need, ids.data()) != ZP_OK) break;
    s->waiting.pop_front();
    r.table = std::move(ids);
    r.seq_len = r.prompt_len;
    r.state = kRunning;
    r.admit_order = s->admit_counter++;
    s->running.push_back(r.id);
    s->plan_prefill.push_back(r.id);
    ++s->stats.admitted;
  }
  assign_slots(s);

  // 3. decide every running request: compress, decode (growing a block if its last is full),
  //    or wait for a slot
  const std::vector<int32_t> order = s->running;
  for (int32_t id : order) {
    Request& r = s->reqs[id];
    if (r.state != kRunning) continue;  // preempted earlier in this loop
    const bool at_cap = static_cast<int32_t>(r.table.size()) >= n_max && r.seq_len >= static_cast<int32_t>(r.table.size()) * b;
    const bool over_cap = r.seq_len > n_max * b;  // left a long prefill
    if (at_cap || over_cap) {
      if (r.has_slot) {
        s->plan_compress.push_back(id);
      } else {
        ++s->stats.slot_waits;
      }
      continue;
    }
    if (s->restricted && !r.has_slot) continue;
    if (r.seq_len == static_cast<int32_t>(r.table.size()) * b && !grow(s, id)) continue;
    s->plan_decode.push_back(id);
  }
  // requests preempted after they were planned do not run
  auto gone = [&](int32_t id) { return s->reqs[id].state != kRunning; };
  s->plan_decode.erase(std::remove_if(s->plan_decode.begin(), s->plan_decode.end(), gone), s->plan_decode.end());
  s->plan_compress.erase(std::remove_if(s->plan_compress.begin(), s->plan_compress.end(), gone),
                         s->plan_compress.end());
  if (s->restricted) ++s->stats.restricted_steps;
  ++s->stats.steps;
  int64_t used = 0;
  for (int32_t id : s->running) used += static_cast<int64_t>(s->reqs[id].table.size());
  s->stats.blocks_in_use = used;
  s->stats.running = static_cast<int32_t>(s->running.size());

  plan->num_decode = static_cast<int32_t>(s->plan_decode.size());
  plan->decode_ids = s->plan_decode.data();
  plan->num_compress = static_cast<int32_t>(s->plan_compress.size());
  plan->compress_ids = s->plan_compress.data();
  plan->num_prefill = static_cast<int32_t>(s->plan_prefill.size());
  plan->prefill_ids = s->plan_prefill.data();
  plan->num_preempted = static_cast<int32_t>(s->plan_preempted.size());
  plan->preempted_ids = s->plan_preempted.data();
  plan->restricted = s->restricted ? 1 : 0;
  return ZP_OK;
}

zp_status zp_sched_request(const zp_sched* s, int32_t id, zp_sched_request_info* info) {
  if (!s || !info || id < 0 || id >= static_cast<int32_t>(s->reqs.size())) return ZP_ERR_INVALID_ARG;
  const Request& r = s->reqs[id];
  info->state = r.state;
  info->seq_len = r.seq_len;
  info->generated = r.generated;
  info->num_blocks = static_cast<int32_t>(r.table.size());
  info->table = r.table.empty() ? nullptr : r.table.data();
  info->has_slot = r.has_slot ? 1 : 0;
  info->preemptions = r.preemptions;
  return ZP_OK;
}

zp_status zp_sched_get_stats(const zp_sched* s, zp_sched_stats* out) {
  if (!s || !out) return ZP_ERR_INVALID_ARG;
  *out = s->stats;
  return ZP_OK;
}

}  // extern "C"
