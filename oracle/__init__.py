"""CPU oracle for GPU-resident tree-speculative greedy decoding with W4A8 verify.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import it.  The
CUDA library never calls into it and shares no code with it.

Sources (cited by page title and section):
* "GPU-Resident Speculative Decoding for In-Browser LLM Inference with WebGPU"
  (research paper): Design > Small-Batch Verification Kernels; Design >
  GPU-Resident Speculation Loop; Design > Draft-Free Drafting From Web Context;
  Design > Feedback Control of Speculation Width; Implementation.
* "WebGPU for LLM Inference, in depth" (blog): "A quantised matrix-vector kernel
  in WGSL" (weight layout, nibble order) and "Worked example: a decode-speed
  budget".
* "Exact Speculative And Assisted Decoding For A Tiny Draft And Qualified
  Champion" (report): section 4 (greedy acceptance, bonus token) and section 7
  (KV commit/rollback as a pointer move).

Floating point is fp64 except where the pages fix a precision (fp32 KV cache,
int8 activation codes, int4 weight codes with 16-bit scales), and except where
a float decides an integer (an activation or weight code): there the oracle
takes the decision in fp32, the precision of the kernels.

Parity unpinned: ``oracle.controller`` (the width controller is a heuristic;
only its decision rule on injected tables is pinned).
"""
