"""CPU oracle for the OSCAR mixed-precision INT2 KV-cache decode path.

TEST INFRASTRUCTURE ONLY. Nothing in the product path may import this
package: only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg
of ``bench.py`` use it. It shares no code, constants or helpers with the CUDA
library; it is written straight from the method's description so that a
reader can check each step against it by eye.

Sources (cited by page title and section throughout):

* the news article "超越 TurboQuant，显存压力终于得到缓解！Together AI 最新论文 OSCAR
  直接挑战 TurboQuant…" (m.youleyou.com), cited as news article "超越 TurboQuant…". Sections used:
  "OSCAR 的出发点", "OSCAR 的设计思路" (token pool, write/read path),
  "精度表现" (bits-per-element budget).
* the MarkTechPost article "Together AI 开源 OSCAR：一种用于长上下文 LLM 服务的注意力感知 2
  位 KV 缓存量化系统" (Chinese translation), cited as MarkTechPost article "Together AI 开源 OSCAR…". Sections
  used: "OSCAR 有何不同做法" (logit-error identity, C_Q, C_S, R_K, R_V,
  Lemma 1, bit reversal), "服务系统：混合精度缓存布局" (S0, W, clipping,
  G_K = 64, per-token asymmetric INT2, R_V absorbed into the projections),
  visual guide step 4 table (c_K, c_V, G_K defaults).

Precision: fp64 everywhere except the quantiser, which is specified op by op
in float32 so that the GPU's codes can be compared bit for bit (a decision
that floating point turns into an integer is taken in the kernel's precision).

Modules:
  rotation  -- calibration statistics, eigenbases, Hadamard, bit reversal, R
  quant     -- clip, per-token asymmetric INT2 quantiser, dequantiser, packing
  pool      -- byte-exact model of the paged mixed-precision token pool
  attention -- exact softmax decode attention and the segmented LSE merge
  projection -- K / V projection (x W^T, rounded to bf16) in front of the write path
"""
from . import rotation, quant, pool, attention, projection  # noqa: F401
