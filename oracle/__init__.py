"""Plain CPU oracle for paged KV-cache decode attention.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path imports, calls or
executes this package: only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may use it.

Every function here is a slow, obviously correct restatement of what the
source pages define, written in NumPy (float64 for attention arithmetic,
IEEE binary32 scalar emulation for the quantiser whose bit pattern must
match the GPU encoder).  It shares no code, header, table or constant
generator with the CUDA library in ``paged_kv_cache_13_gb300``; the two
meet only through the seeded input generators in ``synthetic``.

Sources (cited by page title and section throughout):

* "The 8GB VRAM Breakthrough: How PagedAttention and Dynamic KV-Cache
  Quantization Unlock 64k Context on Consumer GPUs" (a8q9.cn), and its
  Portuguese twin "O Salto dos 8GB de VRAM" (benni-os.net).
* "Capítulo 8 — Gerenciamento de KV Cache de Próxima Geração"
  (LLM Primer VI, actionbridge.io).
* "A Ideia de 60 Anos Que Domou a Memória da GPU" (blog.alisonamorim.com).
* "PagedAttention aplica memória virtual ao cache KV de LLMs"
  (stamatios.com).

Modules:

* ``kv_bytes``   KV-cache size accounting (the KV-cache equation).
* ``allocator``  refcounted free-stack block pool, block tables, fork,
                 copy-on-write append.
* ``attention``  contiguous-slab and paged single-query GQA attention.
* ``quant``      asymmetric INT4 and FP8 E4M3 encoders / decoders.
* ``kvcache``    the KV-append scatter (plain and quantised, with sinks)
                 and the copy-on-write block copy.

Parity status: every function is pinned by a ``-m "not gpu"`` test except
the accuracy of quantised attention against the *original* (unquantised)
data, which the pages only state through perplexity figures that need a
trained model: parity unpinned for that comparison (it is reported, not
asserted).
"""

from . import kv_bytes, allocator, attention, quant, kvcache  # noqa: F401
