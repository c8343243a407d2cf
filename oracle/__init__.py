"""Plain, slow fp64 CPU oracle for page-retrieval sparse attention.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import or call anything in this package.
The product path (the CUDA library and its Python binding) never imports it,
and this package imports nothing from the product.
"""

from .wa_oracle import *  # noqa: F401,F403
