"""Oracle for the radix-cache attention hot path.

TEST INFRASTRUCTURE ONLY.  This package is a plain, slow, obviously correct
CPU restatement of what the pages describe; it exists so that the CUDA library
can be checked against something written independently of it.  Only the
test-suite, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` /
``--impl reference`` legs of ``bench.py`` may import it.  The product path
(``radix_tree_prefix_gb300``) never imports anything from here, and nothing
here imports the product: the two share no code.  Inputs reach the oracle as
plain numpy arrays and Python lists.

Modules
-------
radix_cache  token-granular radix tree + KV slot allocator (match, split,
             lock_ref, leaf-inward cascading heap eviction, insert)
attention    fp64 naive softmax attention (causal extend, decode, LSE merge)
harness      the request flow over the cache (in-batch prefix rule, extend
             batches, decode steps, finish) producing a bookkeeping trace

Parity status of each function is stated in its docstring: every function is
pinned by a ``-m "not gpu"`` test against values the pages print, closed
forms or brute force, except where a docstring says "parity unpinned".
"""
