"""CPU oracle for dynamic block-skipping causal prefill attention.

TEST INFRASTRUCTURE ONLY. Nothing on the product path imports this
package: only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline
leg of ``bench.py`` may call it. It shares no code with the CUDA library.

It is a plain, slow, fp64 restatement of what the method computes, taken
from the dynamic sparse attention deployment guide
("长上下文推理加速方案部署实战：基于动态稀疏注意力机制的推理服务优化指南",
cloud.baidu.com article 9427124), §3.2 "dynamic sparse attention kernel"
and §6.1 "the role of the threshold λ", read as fixed by the design
notes (probability-ratio threshold, per-row test AND-ed over the Q tile).

Modules:

* ``numerics``  -- bf16 / E4M3 decoding and the per-head E4M3 quantiser;
* ``attention`` -- brute-force dense softmax attention (the λ = 0 closed form);
* ``tile_walk`` -- the method: online softmax over 128x128 tiles with the
  skip rule, plus a mask-replay mode that consumes a given skip bitmap;
* ``decisions`` -- a second, non-iterative statement of the skip decisions
  (prefix max of tile row maxima);
* ``layout``    -- the skip-bitmap word layout of the C interface;
* ``importance`` -- the UniPrefill block importance (Eq. 3-4) and top-p
  block selection (§3.3), the second workload on the pages.

Pins (what checks this code against something other than itself) live in
``tests/test_oracle_pins.py`` (attention, skip rule, formats, layout),
``tests/test_oracle_chunked.py`` (query offsets) and
``tests/test_oracle_importance.py`` (block importance, top-p). Every
function is pinned; none is "parity unpinned".
"""
from . import numerics, attention, tile_walk, decisions, layout, importance  # noqa: F401
