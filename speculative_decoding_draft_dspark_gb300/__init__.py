"""GB300-native DSpark draft-and-schedule step: chaining (tcgen05 GEMM with a
fused bias-add + argmax epilogue) and confidence-scheduled verification (one
persistent scheduler kernel), exposed as the C ABI in include/dspark.h."""
from . import dspark  # noqa: F401
from .dspark import *  # noqa: F401,F403

__all__ = [n for n in dir(dspark) if n.startswith("dspark_")]
