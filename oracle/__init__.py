"""The oracle: a plain, slow, obviously correct CPU restatement of what the hot path computes.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline
leg of ``bench.py`` may import anything from here.  The product path (the CUDA library and
its Python binding) never imports, links or runs this package, and this package imports
nothing from the product: the two share no code.  The only module both sides use is the
seeded input generator in ``workloads/``, which holds none of the method's arithmetic.

Contents
--------
radix_tree   radix tree of token ids -> KV-pool slot values: match (with split), insert,
             LRU evict, lock_ref.  Follows the walk-through of SGLang's radix cache
             ("[SGLang] RadixAttention: Radix Tree 기반 프리픽스 캐싱의 핵심").
fp8          OCP FP8 E4M3 ("fn": bias 7, no infinities, max 448) encode/decode, written
             from the OCP 8-bit floating point specification.
kv_store     scatter of new K/V rows into pool slots; bf16 copy or fp8 quantisation.
attention    scaled-dot-product attention per request in float64 (contiguous form and
             the pool-gather form), and the log-sum-exp merge of partial states.
step         the expected outputs of one workload step (every request, or a sample).
schedule     cache-aware ordering of a waiting queue: longest cached prefix first
             ("Efficiently Programming Large Language Models using SGLang" summary,
             §Cache-Aware Scheduling), and first-come-first-served.

Parity pins (tests/test_oracle_*.py) tie each function to something other than itself:
the pages' worked radix example and split example, brute-force tries, torch's independent
float8_e4m3fn cast, pure-Python softmax loops, torch's fp64 SDPA, and closed-form special
cases (constant V, a single key).  No function here is "parity unpinned".
"""
