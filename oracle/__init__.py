"""Float64 CPU oracle (test infrastructure only; see moe_ref)."""
from . import moe_ref  # noqa: F401
