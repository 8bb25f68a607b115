"""fp64 CPU oracle for exact attention (test infrastructure; see ``oracle.attention``)."""
from . import attention  # noqa: F401
