"""Plain, slow, float64 CPU oracle for the per-cycle verify step of MTP speculative decoding.

TEST INFRASTRUCTURE ONLY. Nothing on the product path imports, links or calls this package:
only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline legs of ``bench.py`` may use
it. The CUDA library and its Python binding share no code with it (no kernels, headers, tables
or helpers); the only thing both sides consume is the seeded input generator in ``synth/``,
which holds none of the method's arithmetic. Random numbers the method draws are passed in as
callables or arrays, or generated here from the published Philox definition.

What it follows (sources are the pages' titles and sections):

* lucebox-hub PR #15 "feat(qwen4exp): MTP speculative decoding", sections *What* and
  *Exactness*: draft head over the first 64,000 vocabulary rows with an on-GPU argmax; one
  batched verify of k drafts over k+1 rows; greedy acceptance that emits exactly what decoding
  without drafts emits; rollback that leaves KV and recurrent state bit-identical.
* DS4Server issue #98 "Add Qwen3.8 Flash Next native MTP speculation", sections
  *Implementation* and the closing comment: a draft kept when ``u*q <= p``, a rejection
  replaced by a draw from ``max(0, p - q)``, defined outcomes for zero and non-finite
  probabilities, an EOS among the drafts ending the block, per-verify-row state snapshots,
  rejected rows dropped, a replay fallback.
* llama.cpp PR #28104 "qwen4exp : port NextN/MTP speculative decoding to master", its commits
  on rollback through whole-state checkpoints, on a replay that looped forever, and on keeping
  the checkpoints in device memory: restore, then replay the accepted tokens without checking
  them again, with the state never leaving the device.
* Adaptive verify width (``adapt``; lucebox-hub PR #15, *What* and *Speed*): a per-depth moving
  average of acceptance and a cycle-cost table choose the next width (the controller is this
  build's reading; the pages give none).
* 4-bit affine LM-head weights (``quant``; DS4Server issue #98, closing comment: 4-bit affine
  values in groups of 32): the byte layout and the once-rounded bf16 dequantisation are this
  build's reading.
* Philox4x32-10: Salmon, Moraes, Dror and Shaw, "Parallel Random Numbers: As Easy as 1, 2, 3",
  SC'11, section 3 (the Philox S-box) and Table 2 (round constants).

Modules: ``philox`` (uniforms), ``lmhead`` (logits and row statistics), ``accept`` (drafting,
acceptance, residual and bonus sampling, EOS), ``state`` (KV trim, snapshot commit, replay on
the synthetic recurrent step), ``adapt`` (adaptive width), ``quant`` (4-bit weights). Every
function is pinned by a ``-m "not gpu"`` test against closed forms, brute force, library routines
or published test vectors; each module's docstring lists its pins. A function without one would
say "parity unpinned" in its docstring; none does.
"""

from . import philox, lmhead, accept, state, adapt, quant  # noqa: F401
