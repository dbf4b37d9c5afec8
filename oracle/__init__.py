"""Plain, slow CPU oracle for paged-KV attention — TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline /
reference legs may import or run anything in this package.  The library in
``paged_kv_cache_160_gb300/`` never calls it, and this package never imports the
library: the two share no code.

What it computes, and where the method is stated:

* ``formats``          — exact decoding of stored fp16 / bf16 / e4m3 codes to float64
                         (format definitions; e4m3 is the fp8 KV-cache format named on
                         "PagedAttention: manage the KV cache like virtual memory", §3.1).
* ``paged_attention``  — decode and chunked-prefill attention over a paged cache:
                         the block-table address translation of "Lecture 33 — KV Cache
                         management" §2.2, then plain softmax attention in float64
                         (§2.3 and §8.1 row 1: paging changes addressing only, the
                         arithmetic equals dense attention).
* ``cache_ops``        — KV write into slots and copy-on-write block copies
                         (Lecture 33 §2.4; "PagedAttention ... virtual memory" §3.3).
* ``block_manager``    — free-block FIFO, ref_cnt, append/fork/CoW/free
                         ("PagedAttention ... virtual memory" §3.2–§3.3, Lecture 33 §2.4).
* ``workload``         — the oracle's side of one synthetic step: planning on the model
                         above, stored codes of the synthetic tensors, and the step's write
                         and decode on a subset of its sequences.

Parity status: every function here is pinned by ``tests/test_oracle_*.py`` against
values the pages print, closed forms, library routines on contiguous inputs, or
brute force; none is "parity unpinned".
"""
