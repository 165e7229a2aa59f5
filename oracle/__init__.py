"""Float64 CPU oracle (test infrastructure only; see oracle.triforce)."""

from . import triforce  # noqa: F401
