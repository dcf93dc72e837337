"""CPU oracle for the VeriCache draft -> verify -> accept hot path.

TEST INFRASTRUCTURE ONLY.  Nothing in the library may import or call this
package: only ``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline``
/ reference arm of ``bench.py`` use it.  It shares no code with the CUDA path
(no kernels, headers, helpers, tables or pre-/post-processing); both read
their inputs from the seeded generators in ``synth``.

It is deliberately plain: numpy, fp64 for attention and token scores, and the
exact fp32 operation sequence for the quantiser so that codes can be compared
bit for bit.  Each function cites the passage of the pages it follows; the
pages are

* VeriCache: Turning Lossy KV Cache into Lossless LLM Inference
  (gist.science/paper/2605.17613), "Technical Summary" sections
  Core Algorithm, Key System Innovations, Architecture Support;
* its Korean translation (gist.science/ko/paper/2605.17613), same sections.

The pages fix the loop's semantics but no numeric recipe for the compressors.
The recipe followed here (KIVI-style int2/int4 codes, keys per channel and
values per token in groups of 32, asymmetric min/max with fp16 scale and
zero, round-half-even; SnapKV-style scoring from the last 32 prompt queries
with a 7-wide max-pool, keeping 25% and always the last 32 tokens) is this
library's stated reading of the compressors the Architecture Support section
names (KVzip, KIVI, SnapKV).

Pins: every function here is pinned by ``tests/test_oracle_*.py`` to facts
that do not come from the oracle itself (closed forms, brute force on tiny
inputs, hand-built cases, textbook identities).
"""

from . import kivi, attention, tokendrop, accept, loop  # noqa: F401
