// Continuous-batching scheduler driving the block manager.
//
// Follows "LLM推理引擎深度实战：从PagedAttention到分布式推理部署", sections 3.1
// (iteration-level batching: finished requests leave after every iteration,
// waiting ones join), 3.2 (preemption: the request holding the most pages is
// written to host memory, or shorter sequences are dropped, and restored
// later) and 3.3 (first come, first served), and "大模型推理引擎优化：KV Cache 与
// 连续批处理", sections 三 (ContinuousBatchScheduler: keep running requests,
// fill from the waiting queue while the KV budget allows, stop at the first
// request that does not fit) and 4.1 (chunked prefill mixed with decode).
//
// One step, in order:
//  1. retire requests that produced their last output in the previous step;
//  2. reserve one slot for every decoding request, preempting while the free
//     blocks do not cover them: the largest holder (later arrival on a tie)
//     is swapped to the host pool if it fits there, else the smallest holder
//     is dropped for recompute;
//  3. decode: one slot each, in batch order;
//  4. running requests continue their prompt in chunks bounded by the token
//     budget left (max_tokens minus the decodes) and by the blocks they can
//     still get;
//  5. swapped requests return (arrival order) while their blocks fit and the
//     batch has room; they run from the next step;
//  6. waiting requests are admitted (arrival order) with a first chunk while
//     the batch has room, budget is left and the chunk's blocks fit -- the
//     budget is the block manager's live free count, which each admission
//     lowers;
//  7. if nothing ran while requests are running, one is preempted.
// A request preempted in a step returns in a later one at the earliest.  The
// step that prefills a prompt's last token yields the first output; each
// later step appends the previous output's K/V and yields the next.
#include <algorithm>
#include <deque>
#include <memory>
#include <new>
#include <unordered_map>
#include <vector>

#include "pa_internal.h"

namespace {

enum State { WAITING, PREFILL, DECODE, SWAPPED, FINISHED };

struct Req {
  uint64_t id;
  int32_t prompt, max_new;
  int64_t arrival;
  State state = WAITING, resume = WAITING;
  int32_t prefilled = 0, generated = 0;
  int64_t out_at = -1;
  std::vector<int32_t> host;
  int64_t ctx() const { return prefilled + std::max(0, generated - 1); }
  int32_t held() const { return static_cast<int32_t>((ctx() + PA_BLOCK_SIZE - 1) / PA_BLOCK_SIZE); }
};

int64_t blocks_for(int64_t n) { return (n + PA_BLOCK_SIZE - 1) / PA_BLOCK_SIZE; }

}  // namespace

struct pa_sched {
  pa_alloc* alloc = nullptr;
  int32_t num_blocks = 0, max_batch = 0, max_tokens = 0, host_total = 0;
  std::deque<int32_t> host_free;
  std::vector<Req*> waiting, running, swapped;  // waiting, swapped: arrival order
  std::unordered_map<uint64_t, std::unique_ptr<Req>> reqs;
  int64_t arrivals = 0, iteration = 0;
  std::vector<int32_t> table;  // scratch

  // outputs of the current step
  struct Item {
    uint64_t id;
    int32_t kind, start, len;
  };
  std::vector<Item> items;
  std::vector<int64_t> slots, swap_out, swap_in;
  std::vector<uint64_t> finished, recomputed;

  ~pa_sched() { pa_alloc_destroy(alloc); }

  int32_t free_blocks() const {
    int32_t total = 0, f = 0;
    pa_alloc_stats(alloc, &total, &f, nullptr);
    return f;
  }

  static void insert_by_arrival(std::vector<Req*>& q, Req* r) {
    auto it = std::find_if(q.begin(), q.end(), [r](const Req* x) { return x->arrival > r->arrival; });
    q.insert(it, r);
  }

  void remove_running(Req* r) { running.erase(std::find(running.begin(), running.end(), r)); }

  const std::vector<int32_t>& table_of(uint64_t id) {
    int32_t n = 0;
    int64_t ntok = 0;
    table.resize(num_blocks);
    pa_block_table(alloc, id, table.data(), num_blocks, &n, &ntok);
    table.resize(n);
    return table;
  }

  void preempt() {
    Req* v = *std::max_element(running.begin(), running.end(), [](const Req* a, const Req* b) {
      return a->held() != b->held() ? a->held() < b->held() : a->arrival < b->arrival;
    });
    if (v->held() > static_cast<int32_t>(host_free.size()))
      v = *std::min_element(running.begin(), running.end(), [](const Req* a, const Req* b) {
        return a->held() != b->held() ? a->held() < b->held() : a->arrival > b->arrival;
      });
    const std::vector<int32_t>& tab = table_of(v->id);
    remove_running(v);
    v->out_at = iteration - 1;
    if (tab.size() <= host_free.size()) {
      v->host.clear();
      for (int32_t g : tab) {
        const int32_t h = host_free.front();
        host_free.pop_front();
        v->host.push_back(h);
        swap_out.push_back(g);
        swap_out.push_back(h);
      }
      pa_free_seq(alloc, v->id);
      v->resume = v->state;
      v->state = SWAPPED;
      insert_by_arrival(swapped, v);
    } else {
      pa_free_seq(alloc, v->id);
      v->prefilled = v->generated = 0;
      v->state = WAITING;
      insert_by_arrival(waiting, v);
      recomputed.push_back(v->id);
    }
  }

  int32_t decode_need() const {
    int32_t n = 0;
    for (const Req* r : running)
      if (r->state == DECODE && r->ctx() == static_cast<int64_t>(r->held()) * PA_BLOCK_SIZE) ++n;
    return n;
  }

  void finish_chunk(Req* r) {
    if (r->prefilled == r->prompt) {
      r->state = DECODE;
      r->generated = 1;
      if (r->max_new == 1) r->state = FINISHED;
    }
  }

  void add_item(uint64_t id, int32_t kind, int64_t start, int64_t len) {
    items.push_back({id, kind, static_cast<int32_t>(start), static_cast<int32_t>(len)});
  }

  // Append n tokens to a request's sequence (capacity checked by the caller).
  pa_status append(Req* r, int64_t n) {
    const size_t at = slots.size();
    slots.resize(at + n);
    int64_t s, d;
    return pa_append_tokens(alloc, r->id, n, slots.data() + at, &s, &d);
  }

  pa_status step() {
    items.clear();
    slots.clear();
    swap_out.clear();
    swap_in.clear();
    finished.clear();
    recomputed.clear();
    const int64_t it = iteration++;
    pa_status st;
    // 1. retire
    for (size_t i = 0; i < running.size();) {
      Req* r = running[i];
      if (r->state == FINISHED) {
        pa_free_seq(alloc, r->id);
        running.erase(running.begin() + i);
        finished.push_back(r->id);
        reqs.erase(r->id);
      } else {
        ++i;
      }
    }
    // 2. reserve the decode appends
    while (!running.empty() && decode_need() > free_blocks()) preempt();
    // 3. decodes
    int32_t n_dec = 0;
    for (Req* r : running) {
      if (r->state != DECODE) continue;
      const int64_t start = r->ctx();
      if ((st = append(r, 1)) != PA_OK) return st;
      add_item(r->id, PA_SCHED_DECODE, start, 1);
      if (++r->generated == r->max_new) r->state = FINISHED;
      ++n_dec;
    }
    int64_t budget = std::max<int64_t>(0, static_cast<int64_t>(max_tokens) - n_dec);
    // 4. prefill continuation
    for (Req* r : running) {
      if (r->state != PREFILL || budget == 0) continue;
      const int64_t room = static_cast<int64_t>(r->held()) * PA_BLOCK_SIZE - r->ctx() +
                           static_cast<int64_t>(free_blocks()) * PA_BLOCK_SIZE;
      const int64_t chunk = std::min<int64_t>({r->prompt - r->prefilled, budget, room});
      if (chunk <= 0) continue;
      const int64_t start = r->ctx();
      if ((st = append(r, chunk)) != PA_OK) return st;
      add_item(r->id, PA_SCHED_PREFILL, start, chunk);
      r->prefilled += static_cast<int32_t>(chunk);
      budget -= chunk;
      finish_chunk(r);
    }
    // 5. swapped requests return, in arrival order
    while (!swapped.empty() && static_cast<int32_t>(running.size()) < max_batch) {
      Req* v = swapped.front();
      if (v->out_at == it || blocks_for(v->ctx()) > free_blocks()) break;
      swapped.erase(swapped.begin());
      if ((st = pa_alloc_seq(alloc, v->id, v->ctx())) != PA_OK) return st;
      const std::vector<int32_t>& tab = table_of(v->id);
      for (size_t i = 0; i < tab.size(); ++i) {
        swap_in.push_back(v->host[i]);
        swap_in.push_back(tab[i]);
        host_free.push_back(v->host[i]);
      }
      v->host.clear();
      v->state = v->resume;
      running.push_back(v);
    }
    // 6. admissions, first come first served
    while (!waiting.empty() && static_cast<int32_t>(running.size()) < max_batch && budget > 0) {
      Req* r = waiting.front();
      const int64_t chunk = std::min<int64_t>(r->prompt, budget);
      if (r->out_at == it || blocks_for(chunk) > free_blocks()) break;
      waiting.erase(waiting.begin());
      if ((st = pa_alloc_seq(alloc, r->id, 0)) != PA_OK) return st;
      if ((st = append(r, chunk)) != PA_OK) return st;
      add_item(r->id, PA_SCHED_PREFILL, 0, chunk);
      r->prefilled = static_cast<int32_t>(chunk);
      r->state = PREFILL;
      budget -= chunk;
      finish_chunk(r);
      running.push_back(r);
    }
    // 7. nothing could run: make room for the others
    if (items.empty() && swap_in.empty() && swap_out.empty() && running.size() > 1) preempt();
    return PA_OK;
  }
};

extern "C" {

pa_status pa_sched_create(int32_t num_blocks, const int64_t* free_order, int32_t max_batch, int32_t max_tokens,
                          int32_t host_blocks, pa_sched** out) {
  if (!out) return pa::fail(PA_ERR_INVALID, "pa_sched_create: out is NULL");
  *out = nullptr;
  if (max_batch <= 0 || max_tokens <= 0 || host_blocks < 0)
    return pa::fail(PA_ERR_INVALID, "pa_sched_create: max_batch, max_tokens must be > 0, host_blocks >= 0");
  pa_alloc* a = nullptr;
  pa_status st = pa_alloc_create(num_blocks, PA_BLOCK_SIZE, free_order, &a);
  if (st != PA_OK) return st;
  pa_sched* s = new (std::nothrow) pa_sched();
  if (!s) {
    pa_alloc_destroy(a);
    return pa::fail(PA_ERR_OOM, "pa_sched_create: host allocation failed");
  }
  s->alloc = a;
  s->num_blocks = num_blocks;
  s->max_batch = max_batch;
  s->max_tokens = max_tokens;
  s->host_total = host_blocks;
  for (int32_t i = 0; i < host_blocks; ++i) s->host_free.push_back(i);
  *out = s;
  return pa::ok();
}

void pa_sched_destroy(pa_sched* s) { delete s; }

pa_status pa_sched_add(pa_sched* s, uint64_t id, int32_t prompt_len, int32_t max_new_tokens) {
  if (!s) return pa::fail(PA_ERR_INVALID, "pa_sched_add: null handle");
  if (s->reqs.count(id)) return pa::fail(PA_ERR_INVALID, "pa_sched_add: request id in use");
  if (prompt_len < 1 || max_new_tokens < 1)
    return pa::fail(PA_ERR_INVALID, "pa_sched_add: prompt_len and max_new_tokens must be >= 1");
  if (blocks_for(static_cast<int64_t>(prompt_len) + max_new_tokens) > s->num_blocks)
    return pa::fail(PA_ERR_INVALID, "pa_sched_add: request cannot complete in a pool of %d blocks",
                    s->num_blocks);
  auto r = std::unique_ptr<Req>(new (std::nothrow) Req());
  if (!r) return pa::fail(PA_ERR_OOM, "pa_sched_add: host allocation failed");
  r->id = id;
  r->prompt = prompt_len;
  r->max_new = max_new_tokens;
  r->arrival = s->arrivals++;
  s->waiting.push_back(r.get());
  s->reqs.emplace(id, std::move(r));
  return pa::ok();
}

pa_status pa_sched_step(pa_sched* s, pa_sched_step_out* o) {
  if (!s || !o) return pa::fail(PA_ERR_INVALID, "pa_sched_step: null argument");
  if (!o->ids || !o->kinds || !o->starts || !o->lens || !o->slots || !o->finished || !o->swap_out ||
      !o->swap_in || !o->recomputed)
    return pa::fail(PA_ERR_INVALID, "pa_sched_step: an output array is NULL");
  pa_status st = s->step();
  if (st != PA_OK) return st;
  o->n_items = static_cast<int32_t>(s->items.size());
  for (size_t i = 0; i < s->items.size(); ++i) {
    o->ids[i] = s->items[i].id;
    o->kinds[i] = s->items[i].kind;
    o->starts[i] = s->items[i].start;
    o->lens[i] = s->items[i].len;
  }
  o->n_slots = static_cast<int64_t>(s->slots.size());
  std::copy(s->slots.begin(), s->slots.end(), o->slots);
  o->n_finished = static_cast<int32_t>(s->finished.size());
  std::copy(s->finished.begin(), s->finished.end(), o->finished);
  o->n_swap_out = static_cast<int32_t>(s->swap_out.size() / 2);
  std::copy(s->swap_out.begin(), s->swap_out.end(), o->swap_out);
  o->n_swap_in = static_cast<int32_t>(s->swap_in.size() / 2);
  std::copy(s->swap_in.begin(), s->swap_in.end(), o->swap_in);
  o->n_recomputed = static_cast<int32_t>(s->recomputed.size());
  std::copy(s->recomputed.begin(), s->recomputed.end(), o->recomputed);
  return pa::ok();
}

const pa_alloc* pa_sched_allocator(const pa_sched* s) { return s ? s->alloc : nullptr; }

pa_status pa_sched_limits(const pa_sched* s, int32_t* max_batch, int32_t* max_tokens, int32_t* num_blocks) {
  if (!s || !max_batch || !max_tokens || !num_blocks) return pa::fail(PA_ERR_INVALID, "pa_sched_limits: null argument");
  *max_batch = s->max_batch;
  *max_tokens = s->max_tokens;
  *num_blocks = s->num_blocks;
  return pa::ok();
}

pa_status pa_sched_stats(const pa_sched* s, int32_t* n_waiting, int32_t* n_running, int32_t* n_swapped,
                         int32_t* free_blocks, int32_t* free_host_blocks) {
  if (!s || !n_waiting || !n_running || !n_swapped || !free_blocks || !free_host_blocks)
    return pa::fail(PA_ERR_INVALID, "pa_sched_stats: null argument");
  *n_waiting = static_cast<int32_t>(s->waiting.size());
  *n_running = static_cast<int32_t>(s->running.size());
  *n_swapped = static_cast<int32_t>(s->swapped.size());
  *free_blocks = s->free_blocks();
  *free_host_blocks = static_cast<int32_t>(s->host_free.size());
  return pa::ok();
}

}  // extern "C"
