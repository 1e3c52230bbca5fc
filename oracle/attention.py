"""Paged attention by its definition, in float64 (test infrastructure).

What is computed
----------------
[LLM-INF] section 2.3 states that the paged kernel translates a logical
token index into a physical page through the page table and gathers the
scattered K/V, and that this is transparent to the model computation: the
result is exactly ordinary attention over the sequence's K/V.  So the oracle
is that plain definition, written out:

    for every sequence b and query head h (kv head g = h // G):
        K_t = k_cache[block_tables[b][t // 16], g, t % 16, :]  t < L_b
        V_t = v_cache[ same index ]
        s_t = scale * <q[b, h], K_t>
        out[b, h] = sum_t exp(s_t - max s) V_t / sum_t exp(s_t - max s)

Readings where the pages are silent (each is listed with the design notes):
* the cache layout is [num_blocks, num_kv_heads, 16, head_dim] for K and V;
  16 is the page size printed in [KV-CB] 2.2 and [LLM-INF] 2.2;
* grouped query heads use contiguous groups, kv head = h // (Hq / Hkv);
* context_lens[b] counts the token written in the same decode step;
  a length of 0 gives an all-zero output row;
* FP8 caches hold E4M3 codes (uint8) and INT8 caches signed integer codes
  (int8), with one float32 scale per (block, slot) for K and one for V; the
  stored value is decode(code) * scale (for INT8, code * scale).

No blocking, split or reordering is applied: one softmax per (b, h) over the
whole context, as the definition reads.
"""
import numpy as np

from .fp8_e4m3 import e4m3_decode

BLOCK_SIZE = 16


def _as_f64(x):
    return np.asarray(x).astype(np.float64)


def gather_kv(cache, block_tables_row, n_tokens, kv_head, scales=None):
    """Return float64 [n_tokens, D] of one kv head of one sequence.

    cache: [num_blocks, Hkv, 16, D] array (float16/float32 values, or uint8
    E4M3 / int8 codes when ``scales`` is given); scales: [num_blocks, 16] float32.
    """
    t = np.arange(n_tokens)
    blk = np.asarray(block_tables_row)[t // BLOCK_SIZE].astype(np.int64)
    off = t % BLOCK_SIZE
    rows = cache[blk, kv_head, off, :]
    if scales is None:
        return _as_f64(rows)
    codes = _as_f64(rows) if rows.dtype == np.int8 else e4m3_decode(rows)  # INT8 or E4M3 codes
    return codes * _as_f64(scales)[blk, off][:, None]


def softmax_weights(q_row, K, scale):
    """Normalised softmax weights p_t (float64) of one query over keys K."""
    s = scale * (K @ _as_f64(q_row))
    e = np.exp(s - s.max())
    return e / e.sum()


def paged_decode(q, k_cache, v_cache, block_tables, context_lens, scale,
                 k_scale=None, v_scale=None, heads=None):
    """Paged decode attention, float64 result [B, Hq, D].

    q: [B, Hq, D]; k_cache, v_cache: [num_blocks, Hkv, 16, D];
    block_tables: [B, max_blocks] int; context_lens: [B] int;
    k_scale, v_scale: [num_blocks, 16] float32 for E4M3 caches, else None;
    heads: optional list of (b, h) pairs to evaluate (others stay 0), so
    that large workloads can be checked on a sample.
    """
    q = np.asarray(q)
    B, Hq, D = q.shape
    Hkv = k_cache.shape[1]
    assert Hq % Hkv == 0, "query heads must be a multiple of kv heads"
    G = Hq // Hkv
    out = np.zeros((B, Hq, D), dtype=np.float64)
    wanted = heads if heads is not None else [(b, h) for b in range(B) for h in range(Hq)]
    by_seq = {}
    for b, h in wanted:
        by_seq.setdefault(int(b), []).append(int(h))
    for b, hs in by_seq.items():
        n = int(context_lens[b])
        if n == 0:
            continue
        cache_rows = {}
        for h in hs:
            g = h // G
            if g not in cache_rows:
                cache_rows[g] = (gather_kv(k_cache, block_tables[b], n, g, k_scale),
                                 gather_kv(v_cache, block_tables[b], n, g, v_scale))
            K, V = cache_rows[g]
            p = softmax_weights(q[b, h], K, scale)
            out[b, h] = p @ V
    return out


def paged_prefill(q, q_start, k_cache, v_cache, block_tables, context_lens, scale,
                  k_scale=None, v_scale=None, rows=None):
    """Paged attention for several query tokens per sequence, float64 [T, Hq, D].

    What is computed: [KV-CB] section 4.1 splits a long prompt into chunks
    whose prefill runs beside decode steps, and [LLM-INF] section 6.1 has
    the large model check the draft's gamma tokens in one pass.  Both are
    attention of n_b > 1 new query tokens of sequence b over its paged
    context.  Readings where the pages are silent:

    * the chunk's own K/V are already in the cache (written by the cache
      write beforehand), so context_lens[b] = L_b counts them, and the chunk
      is the last n_b tokens of the context;
    * query token i (0 <= i < n_b) sits at position L_b - n_b + i and sees
      keys 0 .. L_b - n_b + i: the ordinary causal mask, so that splitting a
      prompt into chunks gives the rows a single pass over the whole prompt
      would give;
    * queries are packed: the tokens of sequence b are q[q_start[b] :
      q_start[b+1]]; n_b = 0 is allowed (no rows); a token whose position
      would be negative (n_b > L_b) has no keys and gives a zero row.

    q: [T, Hq, D]; q_start: [B + 1] ints, q_start[0] = 0, nondecreasing;
    other arguments as paged_decode.  rows: optional list of (token, head)
    pairs to evaluate (others stay 0).
    """
    q = np.asarray(q)
    T, Hq, D = q.shape
    Hkv = k_cache.shape[1]
    assert Hq % Hkv == 0, "query heads must be a multiple of kv heads"
    G = Hq // Hkv
    q_start = [int(x) for x in q_start]
    B = len(q_start) - 1
    out = np.zeros((T, Hq, D), dtype=np.float64)
    seq_of = np.zeros(T, dtype=np.int64)
    for b in range(B):
        seq_of[q_start[b]:q_start[b + 1]] = b
    wanted = rows if rows is not None else [(t, h) for t in range(T) for h in range(Hq)]
    by_seq = {}
    for t, h in wanted:
        by_seq.setdefault(int(seq_of[int(t)]), []).append((int(t), int(h)))
    for b, pairs in by_seq.items():
        n = q_start[b + 1] - q_start[b]
        L = int(context_lens[b])
        kv = {}
        for t, h in pairs:
            pos = L - n + (t - q_start[b])
            if pos < 0:
                continue
            g = h // G
            if g not in kv:
                kv[g] = (gather_kv(k_cache, block_tables[b], L, g, k_scale),
                         gather_kv(v_cache, block_tables[b], L, g, v_scale))
            K, V = kv[g]
            p = softmax_weights(q[t, h], K[:pos + 1], scale)
            out[t, h] = p @ V[:pos + 1]
    return out
