"""Oracle for the guided denoise step: a plain, slow CPU restatement in float64.

THIS PACKAGE IS TEST INFRASTRUCTURE.  Only ``tests/``, ``__graft_entry__.smoke()``
and the CPU-baseline / reference legs of ``bench.py`` may import or call it.  The
product path (the CUDA library and its Python binding) never touches it, and it
shares no code, table, constant generator or helper with that path; it does not
import the product package either.  The only module both sides use is the seeded
input generator ``bucketized_guidance_step_gb300.workloads``, which holds random
numbers and rectangles and none of the method's arithmetic.

Sources.  Two web pages define what is computed:

* [SAMPLING] "12 · 采样器、调度器与 CFG" (ComfyUI sampler, scheduler and CFG notes).
  Sections used: "sigma 序列", "denoise 小于 1", "force_full_denoise",
  "CFG 的核心", "cfg = 1 的优化", "calc_cond_batch()：最密集的条件逻辑",
  "为什么要自己拼 batch", "inpaint 与 mask", "一步采样的数据形状".
* [BCG] the write-up on implementing Bucketized Continuous Guidance in SGLang
  (zwxr.cn news 258547).  Sections used: "2. BCG的核心机制拆解",
  "3. 张量并行下的bucket构造", "4. Debug完整链路" (stages 2 and 4).

Where the pages stop (the Karras and "normal" schedules, the Euler update, the
feather profile, the overlap denominator, the inpaint blend, the curve-to-bucket
sampling) each module states the reading it takes and the outside source for it.

Modules:

* ``schedules``  -- sigma schedules, denoise tail, start/last crop, force_full_denoise
* ``buckets``    -- bucket id of a step, curve -> bucket table, per-step scale LUT
* ``step``       -- regional accumulation, guidance combine, inpaint blend, Euler update
* ``mask``       -- bilinear (align_corners=False) pixel-mask -> latent-mask resize
* ``conds``      -- areas to latent slices, packing cond entries into model calls

Every function is pinned by ``tests/test_oracle_*.py`` to closed forms, the
invariants the pages state, library routines or brute force on tiny inputs.
"""

from . import buckets, conds, mask, schedules, step  # noqa: F401
