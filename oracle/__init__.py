"""CPU oracle for speculative-sampling verification.

TEST INFRASTRUCTURE ONLY.  This package is a plain, slow, obviously correct
restatement of what the verification step computes, used to check the CUDA
path.  Only the test suite, ``__graft_entry__.smoke()`` and the CPU-baseline
leg of ``bench.py`` may import it.  The product path (the C-ABI library and
its Python binding) never imports, calls or links anything here, and this
package imports nothing from the product path.

Arithmetic is float64 (numpy) for logit-level inputs.  The probability-level
core (acceptance test, residual, inverse-CDF draw, chain and tree walks) is
written with numpy operations that also work on object arrays of
``fractions.Fraction``, so the same code runs in exact rational arithmetic for
the enumeration pins.

Modules
  philox   counter-based uniforms (Philox4x32-10, Salmon et al., SC'11)
  policy   temperature / top-k / greedy policy -> probability vector
  verify   acceptance, residual, draw, chain walk, tree walk, tree mask

Parity status of each function is given in its docstring; the two readings
the pages leave open and that no page value can pin (the draw's inverse-CDF
order and the uniform keying) are marked "parity unpinned by the pages".
"""

from . import philox, policy, verify  # noqa: F401
