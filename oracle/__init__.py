"""CPU oracle for the routed-MoE forward over int4-grouped experts.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import it.  The
library (``int4_expert_ffn_gb300``) never imports it and shares no code with it.

Parity status of each function (what pins it, see ``tests/test_oracle_pins.py``):

* ``quant_i4g``        pinned: hand-derived bytes in ``tests/golden/``, invariants.
* ``dequant_i4g`` /
  ``matvec_i4g``       pinned: on-grid weights round-trip exactly; numpy matmul.
* ``router_logits`` /
  ``topk``             pinned: brute-force sort, closed-form gates, NaN rule.
* ``topk_sigmoid``     pinned: a hand example with exact sigmoid scores (1/2, 3/4,
                       1/4, 9/10) and closed-form gates, the bias-only-selects
                       rule, invariance to a common bias shift, zero bias picks
                       as softmax, NaN rule.
* ``expert``           pinned: torch float64 SwiGLU on on-grid weights.
* ``moe_forward``      pinned: dense masked MoE, k=1, k=E equal-logit mean,
                       route-count histogram.
* Parity against numbers printed on the pages: unpinned (the pages print no
  worked example of a layer).
"""
from .oracle import *  # noqa: F401,F403
