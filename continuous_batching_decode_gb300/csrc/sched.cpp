// Host-side continuous-batching scheduler: admission with an answer
// reservation and step composition ("20.3 服务、批处理与流式", section 20.3.2
// 批处理, Forma batch mode; FCFS queue from section 20.3.4).
//
// Per plan:
//   1. Admission, first come first served: the queue head is admitted iff a
//      slot is free and free_blocks - sum(outstanding reservations) covers
//      blocks(prompt + min(max_tokens, answer_budget)).  Admission freezes
//      while a row waits for a block.  The lowest free slot is used.
//   2. Prefill chunks first, admission order, min(chunk, prompt left, rows
//      left) rows each; the chunk that completes a prompt samples its last
//      row.
//   3. One decode row per decoding sequence, ordered by (steps waited desc,
//      admission order); a row that needs a block beyond its reservation
//      takes an unreserved free block or waits.  No eviction.
//   4. If no row could be planned while sequences run, the youngest is
//      stopped (or CBD_EDEADLOCK is returned when the fallback is off).
// Blocks come from a min-heap (lowest id first) so plans are reproducible.
//
// Overload and backpressure (section 20.3.4 背压与取消), each off when its
// config field is 0:
//   * bounded admission queue: at most queue_per_slot * max_slots requests
//     wait; a submit beyond that is refused at once (CBD_EBUSY, "busy,
//     retry later");
//   * queue timeout: a request still waiting more than queue_timeout_ms
//     after its submit (caller-driven clock) finishes TIMEOUT before the
//     next admission -- a different outcome from a client cancel;
//   * non-blocking delivery: every request has a buffer of out_buffer
//     undelivered tokens that its client drains (cbd_sched_read); a token
//     that finds the buffer full is not delivered and the request is
//     cancelled (LAGGING), so one slow client never holds up the batch;
//   * abort (client gone): the request stops at once and returns its slot
//     and blocks -- at the commit of a step in flight, whose KV writes
//     still target them.
// The page wakes queued requests with a coalescing capacity signal; here
// admission is re-evaluated in every plan, which sees every release since
// the last one, so no wake-up can be lost.
//
// Second composition policy (cfg.policy == CBD_POLICY_ALBATROSS), after the
// Albatross worker loop ("RWKV Runner Albatross 后端", 连续批处理：Worker 主循环):
// admission also stops while max_prefill requests are prefilling; a prompt
// shorter than short_prompt tokens gets one prefill row per step; a longer
// prompt gets a chunk only in a "sequence step", which comes after every
// prefill_every steps that carried other rows, or at once when there are
// none.  Rows stay prefill-first; the reservation rule is unchanged.
#include <algorithm>
#include <cstring>
#include <deque>
#include <functional>
#include <memory>
#include <queue>
#include <unordered_map>
#include <unordered_set>
#include <vector>

#include "cbd_internal.h"

namespace {

struct Req {
  uint64_t id = 0;
  std::vector<int32_t> prompt;
  int32_t max_tokens = 0;
  cbd_sampling sampling{};
  int32_t slot = -1;
  std::vector<int32_t> blocks;
  int32_t reserved = 0;
  int32_t n_prefilled = 0;
  std::vector<int32_t> generated;
  int64_t waited = 0;
  bool block_wait = false;
  int64_t admit_seq = -1;
  int32_t pending_prefill = 0;
  int64_t arrival_ms = 0;
  bool aborted = false;            // abort requested while a step was in flight
  std::deque<int32_t> outbox;      // delivered, not yet read by the client
};

struct Finished {
  int32_t reason;
  std::vector<int32_t> tokens;
  std::deque<int32_t> outbox;
};

int64_t blocks_for(int64_t positions, int64_t bs) { return (positions + bs - 1) / bs; }

}  // namespace

struct cbd_sched {
  cbd_sched_config cfg{};
  std::priority_queue<int32_t, std::vector<int32_t>, std::greater<int32_t>> free_heap;
  std::vector<Req*> slots;
  std::deque<std::unique_ptr<Req>> waiting;
  std::vector<std::unique_ptr<Req>> running;  // admission order
  std::unordered_map<uint64_t, Finished> finished;
  std::unordered_set<uint64_t> known_ids;
  std::deque<cbd_finished> side_finished;    // finished outside a commit
  int64_t admit_counter = 0;
  int64_t now_ms = 0;
  int32_t seq_countdown = 0;       // Albatross: steps left before the next sequence step
  bool seq_step = false;           // Albatross: the composed step is a sequence step
  bool have_plan = false;
  cbd_sched_stats st{};
  // plan storage
  std::vector<cbd_row> rows;
  std::vector<cbd_sampling> samp;
  std::vector<uint64_t> samp_ids;
  std::vector<int32_t> tables, nblocks, resets;
  std::vector<uint64_t> stopped;

  int32_t free_count() const { return (int32_t)free_heap.size(); }
  int64_t outstanding() const {
    int64_t o = 0;
    for (auto& r : running) o += std::max<int64_t>(0, (int64_t)r->reserved - (int64_t)r->blocks.size());
    return o;
  }
  int32_t need(const Req& r) const {
    if (!cfg.reserve_answer) return 0;
    return (int32_t)blocks_for((int64_t)r.prompt.size() + std::min(r.max_tokens, cfg.answer_budget),
                               cfg.block_size);
  }
  bool grow(Req& r) {
    if (free_heap.empty()) return false;
    if ((int32_t)r.blocks.size() < r.reserved || (int64_t)free_count() - outstanding() > 0) {
      r.blocks.push_back(free_heap.top());
      free_heap.pop();
      return true;
    }
    return false;
  }
  void release(Req* r, int32_t reason) {
    for (int32_t b : r->blocks) free_heap.push(b);
    r->blocks.clear();
    slots[r->slot] = nullptr;
    finished[r->id] = Finished{reason, r->generated, std::move(r->outbox)};
    for (size_t i = 0; i < running.size(); ++i)
      if (running[i].get() == r) {
        running.erase(running.begin() + (ptrdiff_t)i);
        break;
      }
  }
  // Waiters older than the queue timeout leave the queue (reason TIMEOUT).
  void expire() {
    if (cfg.queue_timeout_ms <= 0) return;
    for (size_t i = 0; i < waiting.size();) {
      Req& r = *waiting[i];
      if (now_ms - r.arrival_ms > cfg.queue_timeout_ms) {
        finished[r.id] = Finished{CBD_FINISH_TIMEOUT, {}, {}};
        side_finished.push_back(cbd_finished{r.id, CBD_FINISH_TIMEOUT, 0});
        st.timed_out++;
        waiting.erase(waiting.begin() + (ptrdiff_t)i);
      } else {
        ++i;
      }
    }
  }
  bool albatross() const { return cfg.policy == CBD_POLICY_ALBATROSS; }
  int32_t max_prefill() const {
    return cfg.max_prefill > 0 ? cfg.max_prefill : std::max(cfg.max_slots / 8, 1);   // floor(0.125 slots)
  }
  int32_t prefill_every() const { return cfg.prefill_every > 0 ? cfg.prefill_every : 5; }
  int32_t short_prompt() const { return cfg.short_prompt > 0 ? cfg.short_prompt : 10; }
  void admit() {
    for (auto& r : running)
      if (r->block_wait) return;
    int32_t prefilling = 0;
    for (auto& r : running)
      if (r->n_prefilled < (int32_t)r->prompt.size()) ++prefilling;
    while (!waiting.empty()) {
      if (albatross() && prefilling >= max_prefill()) return;
      int32_t slot = -1;
      for (int32_t s = 0; s < cfg.max_slots; ++s)
        if (!slots[s]) { slot = s; break; }
      if (slot < 0) return;
      Req& head = *waiting.front();
      int32_t nd = need(head);
      if (cfg.reserve_answer && (int64_t)free_count() - outstanding() < nd) return;
      std::unique_ptr<Req> r = std::move(waiting.front());
      waiting.pop_front();
      r->slot = slot;
      r->reserved = nd;
      r->admit_seq = admit_counter++;
      slots[slot] = r.get();
      resets.push_back(slot);
      running.push_back(std::move(r));
      ++prefilling;
    }
  }
  struct Wait { Req* r; bool for_block; };
  void compose(std::vector<Wait>& waits) {
    rows.clear();
    samp.clear();
    samp_ids.clear();
    waits.clear();
    int32_t budget = cfg.max_rows;
    std::unordered_set<Req*> prefilling;
    for (auto& up : running) up->pending_prefill = 0;
    seq_step = false;
    if (albatross()) {
      bool other = false, any_seq = false;     // rows other than sequence chunks; sequence prompts
      for (auto& up : running) {
        const Req& r = *up;
        const int32_t P = (int32_t)r.prompt.size();
        if (r.n_prefilled < P) (P < short_prompt() ? other : any_seq) = true;
        else if (!r.generated.empty() && (int32_t)r.generated.size() < r.max_tokens) other = true;
      }
      seq_step = any_seq && (seq_countdown <= 0 || !other);
    }
    for (auto& up : running) {
      Req& r = *up;
      int32_t P = (int32_t)r.prompt.size();
      if (r.n_prefilled >= P) continue;
      int32_t take = cfg.chunk;
      if (albatross()) {
        if (P < short_prompt()) take = 1;        // one-token prefill, every step
        else if (!seq_step) continue;            // a sequence prompt waits for its step
      }
      if (budget == 0) { waits.push_back({&r, false}); continue; }
      int32_t n = std::min({take, P - r.n_prefilled, budget});
      while ((int64_t)r.blocks.size() * cfg.block_size < (int64_t)r.n_prefilled + n && grow(r)) {}
      n = (int32_t)std::min<int64_t>(n, (int64_t)r.blocks.size() * cfg.block_size - r.n_prefilled);
      if (n <= 0) { waits.push_back({&r, true}); continue; }
      bool done = r.n_prefilled + n == P;
      for (int32_t i = 0; i < n; ++i) {
        int32_t p = r.n_prefilled + i;
        int32_t smp = (done && i == n - 1) ? 1 : 0;
        rows.push_back(cbd_row{r.slot, r.prompt[p], p, 1, smp});
        if (smp) {
          cbd_sampling s = r.sampling;
          s.token_index = 0;
          samp.push_back(s);
          samp_ids.push_back(r.id);
        }
      }
      r.pending_prefill = n;
      prefilling.insert(&r);
      budget -= n;
    }
    std::vector<Req*> dec;
    for (auto& up : running) {
      Req& r = *up;
      if (r.n_prefilled == (int32_t)r.prompt.size() && !prefilling.count(&r) &&
          !r.generated.empty() && (int32_t)r.generated.size() < r.max_tokens)
        dec.push_back(&r);
    }
    std::stable_sort(dec.begin(), dec.end(), [](const Req* a, const Req* b) {
      if (a->waited != b->waited) return a->waited > b->waited;
      return a->admit_seq < b->admit_seq;
    });
    for (Req* rp : dec) {
      Req& r = *rp;
      int32_t pos = (int32_t)r.prompt.size() + (int32_t)r.generated.size() - 1;
      if (budget == 0) { waits.push_back({&r, false}); continue; }
      if ((int64_t)pos >= (int64_t)r.blocks.size() * cfg.block_size && !grow(r)) {
        waits.push_back({&r, true});
        continue;
      }
      rows.push_back(cbd_row{r.slot, r.generated.back(), pos, 0, 1});
      cbd_sampling s = r.sampling;
      s.token_index = (uint32_t)r.generated.size();
      samp.push_back(s);
      samp_ids.push_back(r.id);
      budget -= 1;
    }
  }
};

extern "C" {

cbd_status cbd_sched_create(const cbd_sched_config* cfg, cbd_sched** out) {
  if (!out) return cbd::fail(CBD_EINVAL, "out is NULL");
  *out = nullptr;
  if (!cfg) return cbd::fail(CBD_EINVAL, "cfg is NULL");
  const cbd_sched_config& c = *cfg;
  if (c.n_blocks < 1 || c.block_size < 1 || c.max_slots < 1 || c.max_rows < 1 || c.chunk < 1 ||
      c.answer_budget < 0 || c.max_blocks_per_seq < 1 || c.queue_per_slot < 0 || c.queue_timeout_ms < 0 ||
      c.out_buffer < 0 || c.policy < 0 || c.policy > 1 || c.max_prefill < 0 || c.prefill_every < 0 ||
      c.short_prompt < 0)
    return cbd::fail(CBD_EINVAL, "scheduler config out of range");
  try {
    auto s = std::make_unique<cbd_sched>();
    s->cfg = c;
    for (int32_t b = 0; b < c.n_blocks; ++b) s->free_heap.push(b);
    s->slots.assign(c.max_slots, nullptr);
    *out = s.release();
  } catch (...) {
    return cbd::fail(CBD_ENOMEM, "scheduler allocation failed");
  }
  return CBD_OK;
}

cbd_status cbd_sched_destroy(cbd_sched* s) {
  delete s;
  return CBD_OK;
}

cbd_status cbd_sched_submit(cbd_sched* s, const cbd_request* r) {
  if (!s || !r) return cbd::fail(CBD_EINVAL, "NULL argument");
  const cbd_sched_config& c = s->cfg;
  if (r->prompt_len < 1 || !r->prompt || r->max_tokens < 1)
    return cbd::fail(CBD_EINVAL, "empty prompt or max_tokens < 1");
  if (s->known_ids.count(r->id)) return cbd::fail(CBD_EINVAL, "duplicate request id");
  int64_t total = (int64_t)r->prompt_len + r->max_tokens - 1;
  if (blocks_for(total, c.block_size) > c.max_blocks_per_seq)
    return cbd::fail(CBD_EPOOL, "request longer than max_blocks_per_seq blocks");
  int64_t first = blocks_for((int64_t)r->prompt_len + std::min(r->max_tokens, c.answer_budget), c.block_size);
  if (first > c.n_blocks) return cbd::fail(CBD_EPOOL, "request can never fit the pool");
  if (c.queue_per_slot > 0 && (int64_t)s->waiting.size() >= (int64_t)c.queue_per_slot * c.max_slots) {
    s->st.rejected_busy++;
    return cbd::fail(CBD_EBUSY, "admission queue full; retry later");
  }
  try {
    auto q = std::make_unique<Req>();
    q->id = r->id;
    q->prompt.assign(r->prompt, r->prompt + r->prompt_len);
    q->max_tokens = r->max_tokens;
    q->sampling = r->sampling;
    q->arrival_ms = s->now_ms;
    s->known_ids.insert(r->id);
    s->waiting.push_back(std::move(q));
  } catch (...) {
    return cbd::fail(CBD_ENOMEM, "submit allocation failed");
  }
  return CBD_OK;
}

cbd_status cbd_sched_plan(cbd_sched* s, cbd_plan* out) {
  if (!s || !out) return cbd::fail(CBD_EINVAL, "NULL argument");
  std::memset(out, 0, sizeof(*out));
  const cbd_sched_config& c = s->cfg;
  s->resets.clear();
  s->stopped.clear();
  s->expire();
  s->admit();
  std::vector<cbd_sched::Wait> waits;
  for (;;) {
    s->compose(waits);
    if (!s->rows.empty() || s->running.empty()) break;
    if (!c.stall_fallback) {
      s->have_plan = false;
      return cbd::fail(CBD_EDEADLOCK, "every running sequence is stuck (pool exhausted)");
    }
    Req* young = s->running.front().get();
    for (auto& r : s->running)
      if (r->admit_seq > young->admit_seq) young = r.get();
    s->stopped.push_back(young->id);
    s->st.fallback_stops++;
    s->release(young, CBD_FINISH_FALLBACK);
  }
  if (s->albatross() && !s->rows.empty()) {
    if (s->seq_step) s->seq_countdown = s->prefill_every();
    else s->seq_countdown = std::max(s->seq_countdown - 1, 0);
  }
  std::unordered_set<Req*> w;
  for (auto& x : waits) w.insert(x.r);
  for (auto& r : s->running) {
    if (w.count(r.get())) r->waited++;
    else r->waited = 0;
    r->block_wait = false;
  }
  for (auto& x : waits) x.r->block_wait = x.r->block_wait || x.for_block;
  s->st.stalled_rows += (int64_t)waits.size();

  s->tables.assign((size_t)c.max_slots * c.max_blocks_per_seq, -1);
  s->nblocks.assign(c.max_slots, 0);
  for (auto& r : s->running) {
    for (size_t b = 0; b < r->blocks.size(); ++b)
      s->tables[(size_t)r->slot * c.max_blocks_per_seq + b] = r->blocks[b];
    s->nblocks[r->slot] = (int32_t)r->blocks.size();
  }
  for (auto& row : s->rows) (row.is_prefill ? s->st.rows_prefill : s->st.rows_decode)++;
  if (!s->rows.empty()) s->st.steps++;
  out->n_rows = (int32_t)s->rows.size();
  out->rows = s->rows.data();
  out->n_sampled = (int32_t)s->samp.size();
  out->sampling = s->samp.data();
  out->sampled_ids = s->samp_ids.data();
  out->table_slots = c.max_slots;
  out->block_tables = s->tables.data();
  out->n_blocks_per_slot = s->nblocks.data();
  out->n_resets = (int32_t)s->resets.size();
  out->reset_slots = s->resets.data();
  out->n_stopped = (int32_t)s->stopped.size();
  out->stopped_ids = s->stopped.data();
  s->have_plan = true;
  return CBD_OK;
}

cbd_status cbd_sched_commit(cbd_sched* s, const int32_t* tokens, int32_t m, cbd_finished* fin,
                            int32_t cap, int32_t* n_fin) {
  if (!s) return cbd::fail(CBD_EINVAL, "NULL scheduler");
  if (n_fin) *n_fin = 0;
  if (!s->have_plan) return cbd::fail(CBD_ESTATE, "commit without a plan");
  if (m != (int32_t)s->samp_ids.size()) return cbd::fail(CBD_EINVAL, "token count does not match the plan");
  if (m > 0 && !tokens) return cbd::fail(CBD_EINVAL, "tokens is NULL");
  const int32_t ob = s->cfg.out_buffer;
  std::unordered_map<uint64_t, Req*> by_id;
  for (auto& r : s->running) {
    by_id[r->id] = r.get();
    r->n_prefilled += r->pending_prefill;
    r->pending_prefill = 0;
  }
  // Delivery in row order: a token that finds its request's buffer full is
  // dropped and the request is cancelled (reason LAGGING).
  std::unordered_map<Req*, int32_t> reason;
  for (int32_t j = 0; j < m; ++j) {
    Req* r = by_id.at(s->samp_ids[j]);
    if (r->aborted || reason.count(r)) continue;
    if (ob > 0 && (int32_t)r->outbox.size() >= ob) {
      reason[r] = CBD_FINISH_LAGGING;
      continue;
    }
    r->generated.push_back(tokens[j]);
    if (ob > 0) r->outbox.push_back(tokens[j]);
  }
  int32_t k = 0;
  std::vector<std::pair<Req*, int32_t>> done;
  for (auto& r : s->running) {
    if (r->aborted) done.emplace_back(r.get(), CBD_FINISH_ABORTED);
    else if (reason.count(r.get())) done.emplace_back(r.get(), reason[r.get()]);
    else if ((int32_t)r->generated.size() >= r->max_tokens) done.emplace_back(r.get(), CBD_FINISH_LENGTH);
  }
  for (auto& [r, why] : done) {
    if (fin && k < cap) fin[k] = cbd_finished{r->id, why, (int32_t)r->generated.size()};
    ++k;
    if (why == CBD_FINISH_ABORTED) s->st.aborted++;
    if (why == CBD_FINISH_LAGGING) s->st.lagging++;
    s->release(r, why);
  }
  if (n_fin) *n_fin = std::min(k, cap);
  s->have_plan = false;
  return CBD_OK;
}

cbd_status cbd_sched_abort(cbd_sched* s, uint64_t id) {
  if (!s) return cbd::fail(CBD_EINVAL, "NULL scheduler");
  for (size_t i = 0; i < s->waiting.size(); ++i)
    if (s->waiting[i]->id == id) {
      s->finished[id] = Finished{CBD_FINISH_ABORTED, {}, {}};
      s->side_finished.push_back(cbd_finished{id, CBD_FINISH_ABORTED, 0});
      s->st.aborted++;
      s->waiting.erase(s->waiting.begin() + (ptrdiff_t)i);
      return CBD_OK;
    }
  for (auto& r : s->running)
    if (r->id == id) {
      if (r->aborted) return cbd::fail(CBD_EINVAL, "request already aborted");
      if (s->have_plan) {          // the step in flight still writes its KV blocks
        r->aborted = true;
        return CBD_OK;
      }
      s->side_finished.push_back(cbd_finished{id, CBD_FINISH_ABORTED, (int32_t)r->generated.size()});
      s->st.aborted++;
      s->release(r.get(), CBD_FINISH_ABORTED);
      return CBD_OK;
    }
  return cbd::fail(CBD_EINVAL, "unknown or finished request id");
}

cbd_status cbd_sched_set_time(cbd_sched* s, int64_t now_ms) {
  if (!s) return cbd::fail(CBD_EINVAL, "NULL scheduler");
  if (now_ms < s->now_ms) return cbd::fail(CBD_EINVAL, "the scheduler clock must not go backwards");
  s->now_ms = now_ms;
  return CBD_OK;
}

cbd_status cbd_sched_read(cbd_sched* s, uint64_t id, int32_t* tokens, int32_t cap, int32_t* n) {
  if (!s || !n) return cbd::fail(CBD_EINVAL, "NULL argument");
  if (cap > 0 && !tokens) return cbd::fail(CBD_EINVAL, "tokens is NULL");
  *n = 0;
  std::deque<int32_t>* box = nullptr;
  for (auto& r : s->running)
    if (r->id == id) box = &r->outbox;
  if (!box) {
    auto it = s->finished.find(id);
    if (it != s->finished.end()) box = &it->second.outbox;
  }
  if (!box) {
    for (auto& r : s->waiting)
      if (r->id == id) return CBD_OK;           // queued: nothing generated yet
    return cbd::fail(CBD_EINVAL, "unknown request id");
  }
  int32_t k = 0;
  while (k < cap && !box->empty()) {
    tokens[k++] = box->front();
    box->pop_front();
  }
  *n = k;
  return CBD_OK;
}

cbd_status cbd_sched_finished(cbd_sched* s, cbd_finished* out, int32_t cap, int32_t* n) {
  if (!s || !n) return cbd::fail(CBD_EINVAL, "NULL argument");
  if (cap > 0 && !out) return cbd::fail(CBD_EINVAL, "out is NULL");
  int32_t k = 0;
  while (k < cap && !s->side_finished.empty()) {
    out[k++] = s->side_finished.front();
    s->side_finished.pop_front();
  }
  *n = k;
  return CBD_OK;
}

cbd_status cbd_sched_output(cbd_sched* s, uint64_t id, int32_t* tokens, int32_t cap, int32_t* n) {
  if (!s) return cbd::fail(CBD_EINVAL, "NULL scheduler");
  auto it = s->finished.find(id);
  if (it == s->finished.end()) return cbd::fail(CBD_EINVAL, "request has not finished");
  const auto& t = it->second.tokens;
  if (n) *n = (int32_t)t.size();
  if (tokens)
    for (int32_t i = 0; i < cap && i < (int32_t)t.size(); ++i) tokens[i] = t[i];
  return CBD_OK;
}

cbd_status cbd_sched_stats_get(cbd_sched* s, cbd_sched_stats* out) {
  if (!s || !out) return cbd::fail(CBD_EINVAL, "NULL argument");
  cbd_sched_stats st = s->st;
  st.running = (int32_t)s->running.size();
  st.waiting = (int32_t)s->waiting.size();
  st.free_blocks = s->free_count();
  int64_t alloc = 0, res = 0;
  for (auto& r : s->running) { alloc += (int64_t)r->blocks.size(); res += r->reserved; }
  st.allocated = (int32_t)alloc;
  st.reserved = (int32_t)res;
  st.outstanding = (int32_t)s->outstanding();
  *out = st;
  return CBD_OK;
}

}  // extern "C"
