"""CPU oracle for exact scaled-dot-product attention.  TEST INFRASTRUCTURE ONLY.

This package is the plain, slow, fp64 statement of what the GPU library computes.
Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py`` (its ``cpu_baseline``
leg and its ``--impl reference`` arm) may import, call, link or run anything here.
The product path (``exact_tiled_attention_21_gb300``) never touches it, and the
two share no code: the oracle receives plain numpy arrays and knows nothing of
tiles, TMA, TMEM or bf16 rounding beyond the exact widening of its inputs.

Sources (the three web pages the method is taken from):

* [AIE]  wiki.ai-engineering.at, "Flash Attention" — sections "Das Grundproblem"
  (the naive definition), "Tiling Algorithm", "Lösung: Online Softmax".
* [ZIMA] shop.zimaspace.com, "Wie reduziert Flash Attention den Speicherverkehr
  während der lokalen Inferenz?" — sections on online softmax, kernel fusion
  (scale, mask, normalise, aggregate) and the KV cache.
* [JOHE] johe.ru, "Flash Attention: ускорить attention в 6 раз без потери
  точности" — sections "Введение" (the formula), "Проблема 1" (naive code),
  "Стадии вычисления" (forward pass and recomputed gradients) and
  "Почему это точно?" (the result equals standard attention; only the order of
  operations differs).

Modules:

* ``naive``   — O1: materialised S and P in numpy fp64, forward, backward, decode,
  split-KV decode with log-sum-exp merge.
* ``online``  — O3: the online-softmax recurrence of [AIE] as a pure-Python loop
  over key blocks (small inputs only).
* ``twopass`` — O2: a separate C implementation (``twopass.c``), streaming key
  blocks in fp64 (pass 1: row max and row sum; pass 2: normalised weighted sum).

Every function is pinned by ``tests/test_oracle_pins.py`` (closed forms,
invariants, a library routine, finite differences, hand-derived golden values).
No function is "parity unpinned".
"""
