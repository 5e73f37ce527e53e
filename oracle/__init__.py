"""CPU oracle for one flat ragged paged-attention step: TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` / reference
leg of ``bench.py`` may import this package.  The product path (the C-ABI
library and its Python binding) never imports, calls or links anything here,
and this package never imports the product path.

What it computes (plain definitions, numpy, fp64 for all floating point):

* ``paged_attention.slot_mapping`` / ``kv_write`` / ``gather``: the paged store
  ("P3: native paged-KV continuous-batching sampler", Design / paged.py:
  per-layer [num_blocks, block_size, Hkv, D] K and V, copy-free append that
  scatters into (block, offset), gather to contiguous).
* ``paged_attention.attention``: exact causal softmax attention of every query
  row over its own keys, GQA map q_head // (Hq/Hkv), scale 1/sqrt(D)
  (same page, Design / paged.py "'row' = one SDPA per query row over exactly
  its own keys"; Tensor parallelism / Design "Blocked map q_head // group").
* ``fp8``: the float8_e4m3fn KV cache with per-tensor scales: write codes =
  e4m3(x / s) rounded to nearest (ties to even code), saturating at +-448; read
  value = code * s ("P3: native paged-KV continuous-batching sampler", Review,
  kv_dtype item; "Finish RL Training Faster: Bitwise-Consistent, ...", 4.2).
* ``allocator``: LIFO block allocator with refcounts, all-or-nothing capacity
  growth, read-only shared prefix blocks and the layout check
  (same page, Design / paged.py; Evidence item 4).

Pins (tests marked ``not gpu``): the e4m3 format's fixed points, exhaustive round
trips and ties, and torch's float8_e4m3fn cast as a library cross-check; storage-layout equivalence with a plain
contiguous cache ("Optional paged KV cache (vLLM-style) — v1 design",
Implementation order step 1 and step 3), brute force on tiny inputs, closed
forms, a library cross-check (torch scaled_dot_product_attention in fp64), the
integer examples the P3 page prints (Review, "Pool guard off by one"; Memory
accounting) and a 10,000-event allocator property run (Evidence item 4).
"""
