"""Plain, slow CPU oracle for ResidualAttention over a disaggregated KV cache.

TEST INFRASTRUCTURE.  Nothing in the product path imports, calls, links or runs
anything under ``oracle/``; only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` do.  The oracle shares no code with the CUDA
library: it works on the logical (unpaged) tensors of a workload in fp64 NumPy
(attention) and pure Python (allocator), and every function cites the passage
of the pages it restates.

Modules
  residual_attention  materialised unified cache + textbook softmax (fp64), and
                      the dual-accumulator online-softmax restatement
  allocator           pure-Python model of the paged, refcounted fork allocator
  accounting          closed-form memory / page-count formulas

Pins (tests/test_oracle_*.py, run with ``-m "not gpu"``): hand-derived tiny
cases (tests/golden), plain GQA attention from ``torch.nn.functional.
scaled_dot_product_attention`` when B = 0, single-key and q = 0 closed forms,
RoPE as complex multiplication, linearity of RoPE (disaggregated = merged),
associativity of the value path, shift invariance, the ForkServe page-count
table and the ForkKV memory example.  No function here is "parity unpinned".
"""
