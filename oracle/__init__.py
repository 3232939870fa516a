"""CPU oracle for the streamed NF4 LoRA step.

TEST INFRASTRUCTURE ONLY.  Plain, slow, unfused, resident and unstreamed NumPy code that
states what the GPU path must compute.  Only the tests, ``__graft_entry__.smoke()`` and
the CPU-baseline leg of ``bench.py`` may import it; the product path never does, and
this package shares no code with the CUDA library (they meet only in the seeded input
generator ``synth``).

Modules
  nf4     NF4 codebook, blockwise quantise / dequantise, nibble packing, bf16 rounding
  model   Llama-shaped decoder layer with LoRA: forward, hand-derived backward, loss
  sizes   byte counts of a shard and of the resident tensors (the peak-memory bound)
  optim   AdamW on the adapters, gradient accumulation, several training steps

Every function cites the passage of the pages it follows as
(page title, section).  Where the pages say nothing the reading taken is stated
in the function's docstring.
"""
