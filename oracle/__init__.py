"""Float64 CPU oracle for the sink + short-window KV-cache attention path.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path may import this
package: only ``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` /
``--impl reference`` legs of ``bench.py`` use it.  It shares no code, table or
constant generator with the CUDA library; both sides only share the seeded
input generators in ``synth/``.

Each module states the passage of the LongLive pages it restates:

* ``cache_model``  frame sink + rolling short window (pinned first chunk, fixed
  window of recent chunks) -- LongLive summary page (yunpan.plus), 方法
  §3 高效长推理: 短窗口注意力 and 帧汇聚点.
* ``attention``    exact softmax attention restricted to the visible key set.
* ``fp4``          FP4 KV store: E2M1 codes, 16-element blocks, E4M3 block scale,
  fp32 tensor scale -- LongLive 2.0 inference blog (blog.hotdry.top),
  "NVFP4 量化与 KV Cache 压缩的工程实现" (inference.kv_quant).
* ``recache``      KV recache at a prompt switch: K/V projection, RMSNorm, 3D RoPE
  -- LongLive summary page, 方法 §1 KV 重缓存.

Pins (tests marked ``not gpu``) tie every function to something other than
itself: brute-force loops, closed forms, invariants, exhaustive format tables.
"Parity unpinned" parts are listed where they occur: the 3D RoPE band split and
frequency base are a reading (the pages give none), so parity of RoPE is pinned
to that reading only.
"""

from . import attention, cache_model, fp4, recache  # noqa: F401
