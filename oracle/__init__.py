"""Plain, slow CPU oracle for the routed NVFP4/INT8 linear layer and the Temporal Delta Cache.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path may import, call or link this
package: only ``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` /
``--impl reference`` legs of ``bench.py`` use it.  It shares no code with the CUDA
library under ``int8_mixed_precision_gb300/``; the two meet only through the seeded
input generators in ``synth/`` (which hold none of the method's arithmetic).

Source of the method: "6Bit-Diffusion: Inference-Time Mixed-Precision Quantization for
Video Diffusion Models" (arXiv 2603.18742), as summarised on gist.science (EN, IT, ZH
pages) and chatpaper.ai (authors' abstract).  Each function cites the page and section
it restates.

Modules
-------
formats  E2M1 / E4M3 / bf16 number formats and the block-scale tile layout.
dmpq     Gamma predictor, linear error model and routing, block Hadamard transform,
         NVFP4 and per-token INT8 quantisation, the two quantised GEMMs.
tdc      Temporal Delta Cache (commit / skip / decision) and Purified Delta Refresh.

Parity status
-------------
Every function here is pinned by a ``-m "not gpu"`` test against something other than
itself (closed forms, library routines, brute force, hand-worked fixtures under
``tests/golden/``), including the rounding-boundary margins that decide which elements the
GPU parity tests exempt (``tests/test_oracle_margins.py``).  Parity unpinned: the pages' own
alpha, beta and tau values and their definition of the PDR "outlier ratio" (neither is
printed on the pages); the oracle uses the readings listed in the design notes.
"""
