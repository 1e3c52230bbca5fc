"""Float64 CPU oracle for paged decode attention (test infrastructure only).

This package is the plain, slow, obviously-correct statement of what the
paged-KV hot path computes.  It exists to check the CUDA library and is not
part of the product: only the test-suite, the smoke check in
``__graft_entry__`` and the CPU-baseline leg of ``bench.py`` may import it.
It shares no code with ``paged_kv_cache_191_gb300`` (the CUDA path) and never
imports it.

Modules
-------
fp8_e4m3   OCP FP8 E4M3 ("e4m3fn") decode table and round-to-nearest-even,
           saturate-to-finite encoder.
attention  paged decode attention by the definition softmax(q.K^T.scale).V
           over K/V gathered through a block table, and its multi-token
           form (chunked prefill, speculative verification) with the
           causal mask inside the chunk.
cache_ops  cache write (incl. per-token FP8 quantisation) and block copy.
allocator  host block manager model: FIFO free list, block tables,
           refcounted sharing, fork, copy-on-write on append.

Sources (cited by page title and section):
  [LLM-INF]  "LLM推理引擎深度实战：从PagedAttention到分布式推理部署"
             (ybb.press), sections 2.2 (paging, on-demand allocation,
             copy-on-write), 2.3 (page-table resolution inside the kernel),
             3.2 (preemption), 5.3 (FP8 KV cache), 6.1 (speculative
             decoding: the large model verifies gamma draft tokens in one
             pass).
  [KV-CB]    "大模型推理引擎优化：KV Cache 与连续批处理" (devpress.csdn.net),
             sections 2.2 (16-token blocks), 三 (the Rust block manager
             sketch: block table, free list, refcount, append, free,
             utilisation), 4.1 (chunked prefill mixed with decode) and
             4.2 (copy-on-write for shared blocks).
"""
