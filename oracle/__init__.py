"""CPU oracle for the block-scaled FP8 MoE expert computation.

TEST INFRASTRUCTURE ONLY.  This package is a plain, slow, obviously correct
numpy restatement of what the GPU library computes.  Only the test suite,
``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py`` may
import it.  The CUDA library never calls it, shares no code, header, table or
helper with it, and nothing here imports the CUDA library.

Sources (pages, cited by title and section throughout):

* FlashInfer pull request #4287, "feat(cake_alpha_moe): add optimized
  Blackwell W8A8 expert up/down compute" -- the commit summary, the PR
  description ("Final W8 kernel performance (v46)", "Public contract and
  review fixes") and the review comments.
* SGLang pull request #43556, "Requantize block-FP8 MoE weights to UE8M0 for
  DeepGEMM" -- "Motivation" and "Modifications".
* sglang-glm53-flash-sm120 pull request #13, "SM120 FP8 prefill" --
  description and validation notes.
* The E4M3 format itself is defined by the OCP 8-bit floating point
  specification (OFP8), E2M1 by the OCP Microscaling Formats (MX)
  specification; the pages only name them.

Modules:

* ``numerics`` -- E4M3 codec and BF16 rounding, from their format
  definitions.
* ``moe`` -- quantisers, routing plan, gate/up interleave, UE8M0 requant, the
  forward pass (FP32 emulation) and an FP64 twin used to pin it.
* ``inputs`` -- oracle-side inputs regenerated from the seeded workload
  generator, and the parity metrics (tolerances of the forward).
* ``router`` -- top-k expert selection and route weights from router logits
  (the reading of the companion router the pages name).
* ``w4a8`` -- the E2M1-K32 weight x per-row FP8 activation variant of the
  expert computation (E2M1 codec, K32 and per-row quantisers, the forward and
  an FP64 twin used to pin it).

Pinning status: every function here is pinned by a CPU test under
``tests/`` (exhaustive codec checks, closed forms, brute force on tiny inputs,
invariants, special cases that reduce to torch/numpy routines).  The pages
print no worked numeric example, so no value in the oracle is pinned to a
number printed on the pages.
"""

from . import numerics, moe  # noqa: F401  (``inputs`` needs torch: import it explicitly)
