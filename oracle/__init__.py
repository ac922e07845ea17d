"""CPU oracle for the compressed-KV sparse attention layer — TEST INFRASTRUCTURE.

Plain, slow, obviously correct numpy restatements of what the layer computes,
written from these pages:

* "【#3】ds4.c を読み解く" (qiita, DwarfStar series part 3) — sections 1 (ratio
  schedule), 2 (layer cache), 3 (4096-token prefill chunks), 4 (compressor),
  5 (ratio-4 two lanes and 8-row frontier), 6 (indexer), 7 (mixed attention),
  8 (tail-only RoPE and the compression base);
* "vLLM DeepSeek V4 サポート: 効率的な長文コンテキスト注意機構" — section
  "DeepSeek V4 アテンションアーキテクチャ" (shared K=V with inverse RoPE, c4a /
  c128a window geometry, DSA top-k, 128-token window, 9.62 GiB per 1M tokens).

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline leg
may import this package. The CUDA library never does, and this package imports
nothing from it: the two share no code.

Precision: continuous results (pooled rows, norms, attention outputs) are
computed in fp64 from the exact values of the stored inputs and rounded once to
the storage dtype. The indexer score decides integers (the top-k set), so it is
computed in the precision the pages' CPU reference uses, fp32, in one fixed
operation order that the GPU repeats for every row whose rank is in doubt
(``indexer.index_scores``).

Readings of points the pages leave open are listed in each module's docstring.
Parity pins: every function here is pinned by ``tests/test_oracle_*.py``; see
each test's docstring for what it pins.
"""
