"""CPU oracle for paged KV-cache decode attention.

TEST INFRASTRUCTURE.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import, call
or execute anything in this package.  The product (``paged_kv_cache_173_gb300``)
never imports it, and it never imports the product.

Contents:
  pa_oracle.c       float64 C oracle: locate_kv, reshape_and_cache, decode
  c_oracle.py       ctypes front end of the C oracle
  numpy_oracle.py   a second, loop-by-token statement for tiny brute-force checks
  build.py          gcc build of the C oracle

Every function is pinned by ``tests/test_oracle_pins.py`` against facts the
pages fix (the worked locate_kv example, byte sizes), closed forms,
invariants (identity table == contiguous attention, relabelling physical
blocks, shared prefix == duplicated blocks, ctx = 1 returns V) and an
independent library attention (torch scaled_dot_product_attention in
float64).  No function is left unpinned.
"""
