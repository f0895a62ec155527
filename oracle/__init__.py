"""CPU oracle for the paged MLA KV-cache gather.

TEST INFRASTRUCTURE ONLY. The tests, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg are the only callers. The product library never
imports, links or executes anything in this package, and this package imports
nothing from the product.

- ``oracle.gather``: the per-token C loop (``pmg_oracle.c``) behind ctypes.
- ``oracle.plan``: the page-task enumeration of the per-logical-page mapper,
  written in plain Python from the page's description.
"""
