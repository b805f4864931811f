"""Oracle: a plain, slow, float64 CPU implementation of the Whisper encoder hot path.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path imports, calls or
executes this package; only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may use it.  It
shares no code, table or constant generator with the CUDA library.

Modules
  frontend  log-mel front end: chunking, reflect padding, periodic Hann,
            explicit real DFT, Slaney mel filterbank, log10 / clamp / scale.
  encoder   conv stem, sinusoidal positions, pre-LN transformer layers,
            final LayerNorm.
  fp8       OCP FP8 E4M3 codec and per-tensor absmax scaling.

Sources: the whisper-blaze PyPI page ("Direct Kernel API": LayerNorm eps 1e-5;
feature list: 162 LayerNorms) and showcase site ("The Approach" precision
table; "The Solution" kernel cards; "Learnings": E4M3 saturates at 448).  The
pages name the components but never write out the encoder's equations; where
they are silent each function states the reading it takes (the standard
published Whisper encoder).

Pinning: every function is checked by ``tests/test_oracle_*.py`` against
closed forms, invariants, brute force and independent library special cases.
The end-to-end encoder composition itself is "parity unpinned beyond
composition": no published activations exist, so it is trusted through its
pinned parts plus a whole-layer check against torch's own
TransformerEncoderLayer in float64.
"""
