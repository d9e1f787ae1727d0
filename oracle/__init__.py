"""Plain, slow fp64 CPU oracle for linear-logprob scoring and the three-way compare.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline / reference legs of ``bench.py`` may import this package.  The
product path (the CUDA library and its Python binding) never imports, links or
executes anything here, and this package imports nothing from the product.

It shares no code with the CUDA path: the only common dependency is the seeded
input generator ``synth`` (data only, none of the method's arithmetic).

Modules
-------
``oracle.logprob``  the plain definition  logprob = log_softmax(z / tau)[x]
                    with z = bf16(RMSNorm(h)) . W^T, plus lse and top-1.
``oracle.compare``  per-sequence A/B/C mismatch statistics, k3, TIS weights.
``oracle.processed`` the processed (top-k, then top-p) selected-token logprob.
``oracle.fp8``      the FP8 (e4m3, per-row power-of-two scales) head variant,
                    and the set of its admissible results when the bf16
                    rounding of y is within an implementation's error bound
                    of a rounding midpoint.
``oracle.fp32head`` the FP32 head variant (fp32 y, fp32 W).
``oracle.backward`` the backward of the linear logprob (dL/dy, dL/dW).
``oracle.diag``     extended per-sequence diagnostics: |delta| quantiles,
                    probability MAE, top-1 flips, sequence TIS, K1/K3 sums,
                    ratio error, MIS weights, mean w^2.

Every function cites the page passage it follows.  Pins that tie this oracle to
something other than itself live in ``tests/test_oracle_pins.py`` and
``tests/test_oracle_mutations.py``.  Parity status: every function is pinned
(see those tests); none is "parity unpinned".
"""
from .logprob import (  # noqa: F401
    widen_bf16, round_to_bf16, rmsnorm, logits, lse_stats, oracle_logprob,
    oracle_log_softmax_rows,
)
from .compare import (  # noqa: F401
    OracleError, FLAG_EMPTY, FLAG_BAD_MASK, FLAG_NONFINITE, FLAG_BAD_OFFSETS,
    FLAG_K3_OVERFLOW, PAIRS, oracle_compare, oracle_compare_lenient,
)
from .processed import oracle_processed_logprob, process_head, process_row  # noqa: F401
from .fp8 import (bf16_choices, dequantized_weights, e4m3_round, fp8_scale,  # noqa: F401
                  oracle_logprob_fp8, oracle_logprob_fp8_admissible, quantize_rows)
from .fp32head import oracle_logprob_fp32, rmsnorm_unrounded  # noqa: F401
from .backward import logit_grad, oracle_logprob_backward, rmsnorm_backward  # noqa: F401
from .diag import (  # noqa: F401
    QUANTILES, oracle_diag, oracle_diag_lenient, quantile_linear,
)
