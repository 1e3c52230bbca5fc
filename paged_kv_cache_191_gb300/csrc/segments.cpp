// pa_table_segments: the items of pa_decode_append_segments, from the block
// tables (host only).
//
// Beam search forks a prompt's sequence into beams that share its blocks by
// reference count and copy a shared block only when one of them writes to it
// ("LLM推理引擎深度实战：从PagedAttention到分布式推理部署" 2.2;
// "大模型推理引擎优化：KV Cache 与连续批处理" 4.2).  After reselection the
// beams' tables form a tree: all share the prompt's blocks, siblings share
// their parent's.  Per group and table position j, the members holding the
// same physical block at j form a class -- except that a member is alone at
// and after its last block (the block this step's token is written to) --
// and a segment is a maximal run of positions over which a member's class
// stays the same.  Each segment is listed once, by its lowest member, cut
// into items of at most blocks_per_item blocks; a group's items take partial
// slots 0, 1, ... in the order (owner, position), and the list is sorted
// longest first, so the decode grid dispatches the long items (the
// prompt's) before the short tails and no long item starts last.
#include <stdint.h>

#include <algorithm>
#include <vector>

#include "pa_internal.h"

extern "C" pa_status pa_table_segments(const int32_t* block_tables, int32_t max_blocks, const int32_t* context_lens,
                                       const int32_t* group_start, int32_t n_groups, int32_t blocks_per_item,
                                       int32_t* items, int32_t max_items, int32_t* n_items, int32_t* max_slots) {
  if (!block_tables || !context_lens || !group_start || !n_items || (max_items > 0 && !items))
    return pa::fail(PA_ERR_INVALID, "pa_table_segments: null pointer");
  if (max_blocks <= 0 || n_groups < 0 || blocks_per_item < 1 || blocks_per_item > 64 || max_items < 0)
    return pa::fail(PA_ERR_INVALID, "pa_table_segments: max_blocks, n_groups, blocks_per_item or max_items out of range");
  constexpr int kMax = 8;  // members of one group (4-bit indices, <= 8 MMA columns)
  int32_t count = 0, most = 0;
  for (int32_t k = 0; k < n_groups; ++k) {
    const int32_t first = count;
    const int32_t g0 = group_start[k], M = group_start[k + 1] - g0;
    if (g0 < 0 || M < 0 || M > kMax)
      return pa::fail(PA_ERR_INVALID, "pa_table_segments: group %d has %d members (0..%d)", k, M, kMax);
    int32_t nblk[kMax], last[kMax];
    int32_t P = 0;
    for (int m = 0; m < M; ++m) {
      const int32_t L = context_lens[g0 + m];
      if (L < 0 || L > max_blocks * 16)
        return pa::fail(PA_ERR_INVALID, "pa_table_segments: context length %d of sequence %d out of range", L,
                        g0 + m);
      nblk[m] = (L + 15) / 16;
      last[m] = L > 0 ? (L - 1) / 16 : -1;
      if (nblk[m] > P) P = nblk[m];
    }
    const int32_t* row[kMax];
    for (int m = 0; m < M; ++m) row[m] = block_tables + static_cast<int64_t>(g0 + m) * max_blocks;
    uint32_t prev[kMax] = {0, 0, 0, 0, 0, 0, 0, 0};
    int32_t start[kMax] = {0, 0, 0, 0, 0, 0, 0, 0};
    // emit member m's run [start[m], j) of class c when m owns it
    auto emit = [&](int m, uint32_t c, int32_t j) -> bool {
      if (!c || (c & (~c + 1u)) != (1u << m)) return true;
      uint32_t mlist = 0;
      int nm = 0;
      for (int i = 0; i < M; ++i)
        if (c >> i & 1u) mlist |= static_cast<uint32_t>(i) << (4 * nm++);
      for (int32_t p0 = start[m]; p0 < j; p0 += blocks_per_item) {
        if (count >= max_items) return false;
        const int32_t nb = j - p0 < blocks_per_item ? j - p0 : blocks_per_item;
        int32_t* it = items + 4 * static_cast<int64_t>(count++);
        it[0] = k;
        it[1] = static_cast<int32_t>(mlist);
        it[2] = p0;
        it[3] = static_cast<int32_t>(static_cast<uint32_t>(nb | (nm << 8)) |
                                     (static_cast<uint32_t>(count - 1 - first) << 16));  // the group's next slot
      }
      return true;
    };
    // items come out per owner: run each member over all positions in turn
    for (int m = 0; m < M; ++m) {
      for (int32_t j = 0; j <= P; ++j) {
        uint32_t c = 0;
        if (j < nblk[m]) {
          c = 1u << m;
          if (j < last[m])
            for (int i = 0; i < M; ++i)
              if (i != m && j < last[i] && row[i][j] == row[m][j]) c |= 1u << i;
        }
        if (j == 0 || c != prev[m]) {
          if (j > 0 && !emit(m, prev[m], j))
            return pa::fail(PA_ERR_INVALID, "pa_table_segments: more than max_items (%d) items", max_items);
          start[m] = j;
          prev[m] = c;
        }
      }
    }
    if (count - first > 65535)
      return pa::fail(PA_ERR_INVALID, "pa_table_segments: group %d has %d items", k, count - first);
    most = std::max(most, count - first);
  }
  // longest first, ties in the order listed
  std::vector<int32_t> order(count), sorted(static_cast<size_t>(count) * 4);
  for (int32_t i = 0; i < count; ++i) order[i] = i;
  std::stable_sort(order.begin(), order.end(),
                   [&](int32_t x, int32_t y) { return (items[4 * x + 3] & 0xff) > (items[4 * y + 3] & 0xff); });
  for (int32_t i = 0; i < count; ++i)
    for (int c = 0; c < 4; ++c) sorted[4 * static_cast<size_t>(i) + c] = items[4 * static_cast<size_t>(order[i]) + c];
  std::copy(sorted.begin(), sorted.end(), items);
  *n_items = count;
  if (max_slots) *max_slots = most;
  return PA_OK;
}
