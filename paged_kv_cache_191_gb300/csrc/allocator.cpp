// Host block manager for the paged KV cache.
//
// Follows the block manager of "大模型推理引擎优化：KV Cache 与连续批处理",
// section 三 (fixed 16-token blocks, per-request block table, free pool,
// per-block refcount for shared prefixes, utilisation), with copy-on-write
// per "LLM推理引擎深度实战：从PagedAttention到分布式推理部署", section 2.2.
// Where the page's sketch is incomplete or wrong this implementation takes
// these readings: FIFO free list (take front, release to back, tables
// released in logical order); all-or-nothing errors; release frees a block
// only when its refcount reaches zero; append returns the slot; fork shares a
// table; append into a shared partial block moves the sequence to a fresh
// block and reports the copy; block payloads are never zeroed.
#include <algorithm>
#include <deque>
#include <new>
#include <unordered_map>
#include <vector>

#include "pa_internal.h"

struct pa_alloc {
  struct Seq {
    std::vector<int32_t> blocks;
    int64_t ntok = 0;
    uint64_t mark = 0;  // batch call that last named this sequence (duplicate check)
  };
  int32_t total = 0;
  std::deque<int32_t> free_list;
  std::vector<int32_t> refcount;
  std::unordered_map<uint64_t, Seq> seqs;
  // Scratch of the capacity checks, reused across calls: simulated refcounts
  // of the blocks touched (-1 = untouched) and the list of touched blocks.
  std::vector<int32_t> rc_sim;
  std::vector<int32_t> rc_touched;
  uint64_t batch_mark = 0;

  // Simulated refcount view for one capacity check; reset() restores it.
  struct RcView {
    pa_alloc& a;
    int32_t get(int32_t b) const { return a.rc_sim[b] >= 0 ? a.rc_sim[b] : a.refcount[b]; }
    void set(int32_t b, int32_t v) {
      if (a.rc_sim[b] < 0) a.rc_touched.push_back(b);
      a.rc_sim[b] = v;
    }
    ~RcView() {
      for (int32_t b : a.rc_touched) a.rc_sim[b] = -1;
      a.rc_touched.clear();
    }
  };

  int32_t take() {
    int32_t b = free_list.front();
    free_list.pop_front();
    refcount[b] = 1;
    return b;
  }
  void release(int32_t b) {
    if (--refcount[b] == 0) free_list.push_back(b);
  }
  // Fresh blocks one append to `s` would take, given the simulated refcounts
  // `rc` (decremented where the append would copy a shared block).
  static int need_for_append(const Seq& s, RcView& rc) {
    const int64_t cap = static_cast<int64_t>(s.blocks.size()) * PA_BLOCK_SIZE;
    if (s.ntok < cap) {
      const int32_t last = s.blocks.back();
      const int32_t r = rc.get(last);
      if (r > 1) {
        rc.set(last, r - 1);
        return 1;
      }
      return 0;
    }
    return 1;
  }
  // Apply one append (capacity already checked).
  void apply_append(Seq& s, int64_t* slot, int64_t* src, int64_t* dst) {
    *src = -1;
    *dst = -1;
    const int64_t cap = static_cast<int64_t>(s.blocks.size()) * PA_BLOCK_SIZE;
    if (s.ntok < cap) {
      const int32_t last = s.blocks.back();
      if (refcount[last] > 1) {
        const int32_t fresh = take();
        --refcount[last];
        s.blocks.back() = fresh;
        *src = last;
        *dst = fresh;
      }
    } else {
      s.blocks.push_back(take());
    }
    *slot = static_cast<int64_t>(s.blocks[s.ntok / PA_BLOCK_SIZE]) * PA_BLOCK_SIZE +
            s.ntok % PA_BLOCK_SIZE;
    ++s.ntok;
  }
};

extern "C" {

pa_status pa_alloc_create(int32_t num_blocks, int32_t block_size, const int64_t* free_order,
                          pa_alloc** out) {
  if (!out) return pa::fail(PA_ERR_INVALID, "pa_alloc_create: out is NULL");
  *out = nullptr;
  if (num_blocks <= 0) return pa::fail(PA_ERR_INVALID, "pa_alloc_create: num_blocks must be > 0");
  if (block_size != PA_BLOCK_SIZE)
    return pa::fail(PA_ERR_UNSUPPORTED, "pa_alloc_create: block_size must be 16");
  pa_alloc* a = new (std::nothrow) pa_alloc();
  if (!a) return pa::fail(PA_ERR_OOM, "pa_alloc_create: host allocation failed");
  a->total = num_blocks;
  a->refcount.assign(num_blocks, 0);
  a->rc_sim.assign(num_blocks, -1);
  a->seqs.reserve(1024);
  if (free_order) {
    std::vector<char> seen(num_blocks, 0);
    for (int32_t i = 0; i < num_blocks; ++i) {
      const int64_t b = free_order[i];
      if (b < 0 || b >= num_blocks || seen[b]) {
        delete a;
        return pa::fail(PA_ERR_INVALID, "pa_alloc_create: free_order is not a permutation");
      }
      seen[b] = 1;
      a->free_list.push_back(static_cast<int32_t>(b));
    }
  } else {
    for (int32_t i = 0; i < num_blocks; ++i) a->free_list.push_back(i);
  }
  *out = a;
  return pa::ok();
}

void pa_alloc_destroy(pa_alloc* a) { delete a; }

pa_status pa_alloc_seq(pa_alloc* a, uint64_t seq_id, int64_t num_tokens) {
  if (!a) return pa::fail(PA_ERR_INVALID, "pa_alloc_seq: null handle");
  if (num_tokens < 0) return pa::fail(PA_ERR_INVALID, "pa_alloc_seq: negative token count");
  if (a->seqs.count(seq_id)) return pa::fail(PA_ERR_INVALID, "pa_alloc_seq: sequence exists");
  const int64_t need = (num_tokens + PA_BLOCK_SIZE - 1) / PA_BLOCK_SIZE;
  if (need > static_cast<int64_t>(a->free_list.size()))
    return pa::fail(PA_ERR_OOM, "pa_alloc_seq: need %lld blocks, %zu free",
                    static_cast<long long>(need), a->free_list.size());
  pa_alloc::Seq s;
  s.ntok = num_tokens;
  s.blocks.reserve(static_cast<size_t>(need));
  for (int64_t i = 0; i < need; ++i) s.blocks.push_back(a->take());
  a->seqs.emplace(seq_id, std::move(s));
  return pa::ok();
}

pa_status pa_append_slot(pa_alloc* a, uint64_t seq_id, int64_t* slot, int64_t* cow_src,
                         int64_t* cow_dst) {
  if (!a || !slot || !cow_src || !cow_dst)
    return pa::fail(PA_ERR_INVALID, "pa_append_slot: null argument");
  auto it = a->seqs.find(seq_id);
  if (it == a->seqs.end()) return pa::fail(PA_ERR_NOT_FOUND, "pa_append_slot: unknown sequence");
  {
    pa_alloc::RcView rc{*a};
    if (pa_alloc::need_for_append(it->second, rc) > static_cast<int>(a->free_list.size()))
      return pa::fail(PA_ERR_OOM, "pa_append_slot: no free block");
  }
  a->apply_append(it->second, slot, cow_src, cow_dst);
  return pa::ok();
}

pa_status pa_append_slots(pa_alloc* a, const uint64_t* seq_ids, int32_t n, int64_t* slots,
                          int64_t* cow_pairs, int32_t* n_cow) {
  if (!a || n < 0 || (n > 0 && (!seq_ids || !slots || !cow_pairs)) || !n_cow)
    return pa::fail(PA_ERR_INVALID, "pa_append_slots: bad argument");
  std::vector<pa_alloc::Seq*> ss(static_cast<size_t>(n));
  const uint64_t mark = ++a->batch_mark;
  for (int32_t i = 0; i < n; ++i) {
    auto it = a->seqs.find(seq_ids[i]);
    if (it == a->seqs.end())
      return pa::fail(PA_ERR_NOT_FOUND, "pa_append_slots: unknown sequence at %d", i);
    if (it->second.mark == mark)
      return pa::fail(PA_ERR_INVALID, "pa_append_slots: duplicate sequence at %d", i);
    it->second.mark = mark;
    ss[i] = &it->second;
  }
  int64_t need = 0;
  {
    pa_alloc::RcView rc{*a};
    for (int32_t i = 0; i < n; ++i) need += pa_alloc::need_for_append(*ss[i], rc);
  }
  if (need > static_cast<int64_t>(a->free_list.size()))
    return pa::fail(PA_ERR_OOM, "pa_append_slots: need %lld blocks, %zu free",
                    static_cast<long long>(need), a->free_list.size());
  int32_t nc = 0;
  for (int32_t i = 0; i < n; ++i) {
    int64_t src, dst;
    a->apply_append(*ss[i], &slots[i], &src, &dst);
    if (src >= 0) {
      cow_pairs[2 * nc] = src;
      cow_pairs[2 * nc + 1] = dst;
      ++nc;
    }
  }
  *n_cow = nc;
  return pa::ok();
}

pa_status pa_fork(pa_alloc* a, uint64_t parent, uint64_t child) {
  if (!a) return pa::fail(PA_ERR_INVALID, "pa_fork: null handle");
  auto it = a->seqs.find(parent);
  if (it == a->seqs.end()) return pa::fail(PA_ERR_NOT_FOUND, "pa_fork: unknown parent");
  if (a->seqs.count(child)) return pa::fail(PA_ERR_INVALID, "pa_fork: child exists");
  pa_alloc::Seq c = it->second;
  for (int32_t b : c.blocks) ++a->refcount[b];
  a->seqs.emplace(child, std::move(c));
  return pa::ok();
}

pa_status pa_append_tokens(pa_alloc* a, uint64_t seq_id, int64_t n, int64_t* slots,
                           int64_t* cow_src, int64_t* cow_dst) {
  if (!a || n < 0 || !cow_src || !cow_dst)
    return pa::fail(PA_ERR_INVALID, "pa_append_tokens: bad argument");
  auto it = a->seqs.find(seq_id);
  if (it == a->seqs.end()) return pa::fail(PA_ERR_NOT_FOUND, "pa_append_tokens: unknown sequence");
  pa_alloc::Seq& s = it->second;
  *cow_src = -1;
  *cow_dst = -1;
  if (n == 0) return pa::ok();
  // fresh blocks: one copy-on-write for a shared partial last block, plus
  // whatever the n tokens need beyond the current capacity
  const int64_t cap = static_cast<int64_t>(s.blocks.size()) * PA_BLOCK_SIZE;
  int64_t need = 0;
  if (s.ntok < cap) {
    pa_alloc::RcView rc{*a};
    need = pa_alloc::need_for_append(s, rc);
  }
  const int64_t beyond = s.ntok + n - cap;
  if (beyond > 0) need += (beyond + PA_BLOCK_SIZE - 1) / PA_BLOCK_SIZE;
  if (need > static_cast<int64_t>(a->free_list.size()))
    return pa::fail(PA_ERR_OOM, "pa_append_tokens: need %lld blocks, %zu free",
                    static_cast<long long>(need), a->free_list.size());
  for (int64_t i = 0; i < n; ++i) {
    int64_t slot, src, dst;
    a->apply_append(s, &slot, &src, &dst);
    if (slots) slots[i] = slot;
    if (src >= 0) {
      *cow_src = src;
      *cow_dst = dst;
    }
  }
  return pa::ok();
}

pa_status pa_fork_seqs(pa_alloc* a, const uint64_t* parents, const uint64_t* children, int32_t n) {
  if (!a || n < 0 || (n > 0 && (!parents || !children)))
    return pa::fail(PA_ERR_INVALID, "pa_fork_seqs: bad argument");
  {
    // validate: parents exist (or are children made earlier in the batch),
    // children are new and distinct
    std::vector<uint64_t> made(children, children + n);
    std::sort(made.begin(), made.end());
    for (int32_t i = 0; i + 1 < n; ++i)
      if (made[i] == made[i + 1]) return pa::fail(PA_ERR_INVALID, "pa_fork_seqs: repeated child");
    for (int32_t i = 0; i < n; ++i) {
      if (a->seqs.count(children[i]))
        return pa::fail(PA_ERR_INVALID, "pa_fork_seqs: child exists at %d", i);
      if (!a->seqs.count(parents[i])) {
        bool earlier = false;
        for (int32_t k = 0; k < i && !earlier; ++k) earlier = children[k] == parents[i];
        if (!earlier) return pa::fail(PA_ERR_NOT_FOUND, "pa_fork_seqs: unknown parent at %d", i);
      }
    }
  }
  for (int32_t i = 0; i < n; ++i) {
    pa_alloc::Seq c = a->seqs.find(parents[i])->second;
    for (int32_t b : c.blocks) ++a->refcount[b];
    a->seqs.emplace(children[i], std::move(c));
  }
  return pa::ok();
}

pa_status pa_free_seqs(pa_alloc* a, const uint64_t* ids, int32_t n) {
  if (!a || n < 0 || (n > 0 && !ids)) return pa::fail(PA_ERR_INVALID, "pa_free_seqs: bad argument");
  const uint64_t mark = ++a->batch_mark;
  std::vector<decltype(a->seqs.begin())> its(static_cast<size_t>(n));
  for (int32_t i = 0; i < n; ++i) {
    auto it = a->seqs.find(ids[i]);
    if (it == a->seqs.end()) return pa::fail(PA_ERR_NOT_FOUND, "pa_free_seqs: unknown sequence at %d", i);
    if (it->second.mark == mark) return pa::fail(PA_ERR_INVALID, "pa_free_seqs: duplicate sequence at %d", i);
    it->second.mark = mark;
    its[i] = it;
  }
  for (int32_t i = 0; i < n; ++i) {
    for (int32_t b : its[i]->second.blocks) a->release(b);
    a->seqs.erase(its[i]);
  }
  return pa::ok();
}

pa_status pa_reselect(pa_alloc* a, const uint64_t* ids, const int32_t* parent_idx, int32_t n) {
  if (!a || n < 0 || (n > 0 && (!ids || !parent_idx)))
    return pa::fail(PA_ERR_INVALID, "pa_reselect: bad argument");
  const uint64_t mark = ++a->batch_mark;
  std::vector<pa_alloc::Seq*> ss(static_cast<size_t>(n));
  for (int32_t i = 0; i < n; ++i) {
    auto it = a->seqs.find(ids[i]);
    if (it == a->seqs.end()) return pa::fail(PA_ERR_NOT_FOUND, "pa_reselect: unknown sequence at %d", i);
    if (it->second.mark == mark) return pa::fail(PA_ERR_INVALID, "pa_reselect: duplicate sequence at %d", i);
    it->second.mark = mark;
    ss[i] = &it->second;
  }
  for (int32_t i = 0; i < n; ++i)
    if (parent_idx[i] < 0 || parent_idx[i] >= n)
      return pa::fail(PA_ERR_INVALID, "pa_reselect: parent index out of range at %d", i);
  // every new table shares its parent's blocks before any old table is released
  std::vector<std::vector<int32_t>> tabs(static_cast<size_t>(n));
  std::vector<int64_t> ntok(static_cast<size_t>(n));
  for (int32_t i = 0; i < n; ++i) {
    tabs[i] = ss[parent_idx[i]]->blocks;
    ntok[i] = ss[parent_idx[i]]->ntok;
    for (int32_t b : tabs[i]) ++a->refcount[b];
  }
  for (int32_t i = 0; i < n; ++i) {
    for (int32_t b : ss[i]->blocks) a->release(b);
    ss[i]->blocks.swap(tabs[i]);
    ss[i]->ntok = ntok[i];
  }
  return pa::ok();
}

pa_status pa_free_seq(pa_alloc* a, uint64_t seq_id) {
  if (!a) return pa::fail(PA_ERR_INVALID, "pa_free_seq: null handle");
  auto it = a->seqs.find(seq_id);
  if (it == a->seqs.end()) return pa::fail(PA_ERR_NOT_FOUND, "pa_free_seq: unknown sequence");
  for (int32_t b : it->second.blocks) a->release(b);
  a->seqs.erase(it);
  return pa::ok();
}

pa_status pa_block_table(const pa_alloc* a, uint64_t seq_id, int32_t* out, int32_t cap,
                         int32_t* n_blocks, int64_t* n_tokens) {
  if (!a || !n_blocks || !n_tokens || cap < 0 || (cap > 0 && !out))
    return pa::fail(PA_ERR_INVALID, "pa_block_table: bad argument");
  auto it = a->seqs.find(seq_id);
  if (it == a->seqs.end()) return pa::fail(PA_ERR_NOT_FOUND, "pa_block_table: unknown sequence");
  const auto& blocks = it->second.blocks;
  const int32_t nb = static_cast<int32_t>(blocks.size());
  for (int32_t i = 0; i < nb && i < cap; ++i) out[i] = blocks[i];
  *n_blocks = nb;
  *n_tokens = it->second.ntok;
  return pa::ok();
}

pa_status pa_block_tables(const pa_alloc* a, const uint64_t* seq_ids, int32_t n, int32_t* tables,
                          int32_t cap, int32_t* context_lens) {
  if (!a || n < 0 || cap <= 0 || (n > 0 && (!seq_ids || !tables || !context_lens)))
    return pa::fail(PA_ERR_INVALID, "pa_block_tables: bad argument");
  for (int32_t i = 0; i < n; ++i) {
    auto it = a->seqs.find(seq_ids[i]);
    if (it == a->seqs.end())
      return pa::fail(PA_ERR_NOT_FOUND, "pa_block_tables: unknown sequence at %d", i);
    if (static_cast<int64_t>(it->second.blocks.size()) > cap)
      return pa::fail(PA_ERR_INVALID, "pa_block_tables: table of sequence %d exceeds cap", i);
    if (it->second.ntok > INT32_MAX)
      return pa::fail(PA_ERR_INVALID, "pa_block_tables: token count exceeds int32");
  }
  for (int32_t i = 0; i < n; ++i) {
    const auto& s = a->seqs.find(seq_ids[i])->second;
    int32_t* row = tables + static_cast<size_t>(i) * cap;
    const int32_t nb = static_cast<int32_t>(s.blocks.size());
    for (int32_t j = 0; j < cap; ++j) row[j] = j < nb ? s.blocks[j] : -1;
    context_lens[i] = static_cast<int32_t>(s.ntok);
  }
  return pa::ok();
}

pa_status pa_alloc_stats(const pa_alloc* a, int32_t* total, int32_t* free_blocks,
                         int32_t* refcounts) {
  if (!a || !total || !free_blocks) return pa::fail(PA_ERR_INVALID, "pa_alloc_stats: bad argument");
  *total = a->total;
  *free_blocks = static_cast<int32_t>(a->free_list.size());
  if (refcounts)
    for (int32_t i = 0; i < a->total; ++i) refcounts[i] = a->refcount[i];
  return pa::ok();
}

pa_status pa_free_list(const pa_alloc* a, int32_t* out, int32_t cap, int32_t* n) {
  if (!a || !n || cap < 0 || (cap > 0 && !out))
    return pa::fail(PA_ERR_INVALID, "pa_free_list: bad argument");
  int32_t i = 0;
  for (int32_t b : a->free_list) {
    if (i < cap) out[i] = b;
    ++i;
  }
  *n = i;
  return pa::ok();
}

}  // extern "C"
