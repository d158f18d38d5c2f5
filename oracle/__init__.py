"""CPU oracle for position-split, quantised-KV decode attention.

TEST INFRASTRUCTURE ONLY.  Only the test suite, the package entry point's smoke
check and the benchmark's CPU-baseline leg may import this package.  The product
path (the CUDA library and its Python binding) never imports, calls or links it,
and this package never imports the product path.

Plain, slow, obviously-correct NumPy:
  * attention and the LSE combine in float64;
  * the two encoders (q8_0, TurboQuant-MSE 3-bit) as step-by-step IEEE float32
    emulation in a fixed operation order, so that quantised codes can be compared
    bit for bit;
  * the Lloyd-Max codebook solved in float64 from the Gaussian density.

Every function cites the page and section it follows.  Where the pages leave a step
open, the docstring states the reading taken.

Parity status: every function here is pinned by the CPU tests (closed forms,
published tables, library routines, brute force on tiny inputs).  The attention
values themselves have no printed worked example on the pages; they are pinned by
invariants, closed forms and library routines instead.
"""

from . import q8_0, turboquant, attention, pipeline  # noqa: F401
