"""CPU oracle for the MoE-FFN forward layer -- TEST INFRASTRUCTURE ONLY.

A plain, slow, float64 NumPy restatement of what the layer computes, used to
check the CUDA path.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import it.  The product library never
calls it and shares no code with it.

Pages cited (by title; section numbers are the ones printed in each page):
  [P1] «大模型MoE架构揭秘：如何用2%参数实现万亿级算力调度» (mhpn.cn)
  [P2] «项目概述：为什么MoE成了大模型突围的“秘密武器”» (mooersco.com)
  [P3] «DeepSeek-V2: A Strong, Economical, and Efficient Mixture-of-Experts
       Language Model» — paper summary page (wzjinhao.cn)
  [P4] «GPT-4 Has 1.8 Trillion Parameters. It Uses 2% of Them Per Token.» —
       rebuttal page (l189.com)
  [P5] «为什么MoE有效？稀疏激活的数学直觉与工程实践» (ai.learningdata.cn)

Parity status per function is listed in ``moe_oracle.PINS``.
"""
from .moe_oracle import *  # noqa: F401,F403
from .moe_oracle import PINS  # noqa: F401
