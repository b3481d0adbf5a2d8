"""fp64 CPU oracle for the absorbed-MLA decode path.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path imports, calls or
links this package: only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` use it.  It
shares no code with the CUDA library (``mla_latent_kv_uk_gb300/csrc``) and
imports nothing from it.

Each function is the plain definition of one step, written in float64 with
numpy; no blocking, fusion or reordering beyond the definition.  Citations
name the source page by title and the section on it:

* "MLA DCP query replication digest" — prhub digest of vLLM PR 45964,
  一句话：MLA DCP 中通过 query 复制跳过 all-gather 通信
* "DCP + FP8 KV MLA decode digest" — prhub digest of vLLM PR 44044,
  一句话：支持 DCP + FP8 KV Cache 在 MLA 解码中协同
* "PCP+DCP sparse MLA digest" — prhub digest of vLLM PR 56157
* "MLA DCP prefill blog" — DeepSeek MLA 在 DCP 分布式环境中的 Prefill 阶段解析

Every function here is pinned by a ``-m "not gpu"`` test against something
other than itself (closed forms, brute-force scalar loops, identities the
pages fix, library routines); none is "parity unpinned".
"""

from . import codecs, mla  # noqa: F401
