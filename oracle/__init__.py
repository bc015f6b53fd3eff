"""CPU oracle of the speculative-decoding verify step.

TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check of ``__graft_entry__`` and
the CPU-baseline leg of ``bench.py`` may import this package.  The product path (the
CUDA library and its Python binding) never imports, calls or falls back to it, and it
shares no code with that path: the only common module is ``synth`` (seeded inputs).

Everything is plain numpy in float64, written in the order the write-ups describe the
method, so that a reader can check it by eye:

* ``verify``   -- truncation (temperature, top-k, top-p), greedy acceptance, the
                  rejection-sampling acceptance rule with its residual resample, and
                  inverse-CDF sampling.
* ``model``    -- the dense decoder forward (RMSNorm, RoPE, causal GQA attention,
                  SwiGLU) with a per-token KV list that is trimmed by slicing.
* ``generate`` -- plain and speculative generation loops, the scripted and n-gram
                  drafters' definitions.
* ``brute``    -- exact laws of the acceptance rule by enumeration on tiny vocabularies.

Sources (pages of the write-ups, by title and section):
  [SD-Apple]  "Speculative Decoding on Apple Silicon: 119% Faster on Qwen3.8",
              sections "How speculative decoding works", "Why this needed a patch to
              mlx_lm at all".
  [OptiQ]     "Speculative decoding on Apple Silicon" (mlx-optiq docs), sections
              "N-gram lookup: any model", "MTP head", "About depth".
  [MTP-fixes] "Qwen3.5 and Qwen3.6 MTP head reaches 1.4x on Apple Silicon after three
              fixes", sections "The verify was wrong under sampling", "Truncation has to
              match on both sides".
  [Draft]     "What is Speculative Decoding and How Does a Draft Model Work?", sections
              "#2 - A draft model guesses...", "#3 - The output is the same...".

Parity status per function is listed in each module's header.
"""
