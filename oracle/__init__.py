"""fp64 CPU oracle of the text-diffusion canvas sampler -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline / reference legs of
``bench.py`` may import this package. The product path (the CUDA library and its Python
binding) never imports, links or executes anything here, and this package never imports
the product path: the two share no code. Both take their inputs from the seeded generators
in ``canvas_sampler_gb300.workloads``, which hold none of the method's arithmetic.

What is computed, and from which passage (page title, then section):

* logits, full-precision softmax over the vocabulary, self-conditioning vector
  s = softmax(logits / T) . E -- "DiffusionGemma Technical Report", section 6, "Sampling";
  the self-conditioning state fed back into the next pass -- same report, section 8,
  "Finetuning procedure" (z_t from a previous forward pass, z_t = 0 otherwise).
* canvas of 256 uniformly random tokens, refined for at most 48 steps; accepted tokens
  kept, all others re-noised uniformly at random -- "DiffusionGemma: Google's open diffusion
  LLM", section "A diffusion language model refines 256 tokens in 12 steps"; uniform-state
  (multinomial) diffusion -- same article, "Tokens stay editable within a canvas, then freeze";
  confident tokens locked, the rest re-noised -- "Google DeepMind's DiffusionGemma Generates
  Text 4x Faster by Ditching Tokens", "How text diffusion actually works".
* top-k truncation applied to the sampling step only -- technical report section 6,
  "Multi-user throughput".
* Philox4x32-10 -- Salmon, Moraes, Dror and Shaw, "Parallel random numbers: as easy as
  1, 2, 3", SC'11 (the pages name no generator; a counter-based one makes every draw a
  pure function of (seed, sequence, position, token, step)).

Where the pages leave a step open (there is no printed sampler listing in them), the
readings taken are written next to the code that takes them.

Pins (tests/test_oracle_*.py check this package against things other than itself):
closed forms (uniform softmax, s -> E[j] for H = alpha E[j], T -> 0 argmax), brute force
with math.fsum on tiny vocabularies, invariants (probabilities sum to 1, entropy in
[0, ln V], locked tokens never change, >= 1 lock per step, termination), a hand-derived
worked example under tests/golden/, chi-squared tests of Gumbel-max frequencies and of
re-noise uniformity, and for Philox an implementation written by others (the header-only
Philox4x32-10 engine of PyTorch's C++ headers, compiled into a small driver and compared block
for block), a second, scalar implementation, bijectivity and statistical tests.
"""
from .philox import philox4x32_10, philox4x32_10_scalar  # noqa: F401
from .sampler import (  # noqa: F401
    bf16_bits_to_f64,
    f64_to_bf16_bits,
    gumbel_uniforms,
    renoise_tokens,
    softmax_stats,
    sampler_step,
    lock_update,
    entropy_budget_update,
    scheduled_temperature,
    LOCK_THRESHOLD,
    LOCK_ENTROPY_BUDGET,
    standin_hidden,
    denoise_loop,
    block_loop,
)
from .shards import merge_shards, shard_partial  # noqa: F401
