"""GB300-native (sm_103a) per-layer MoE expert path of Specter's Streamlined
Execution Engine: routing, expert-activation counters, gather by expert, the
fused INT4 draft MLP, the expert-reordered FP16 verify MLP, the shared expert
and the weighted combine, as hand-written CUDA behind the C ABI in
include/spx.h (libspx.so).  ``spx`` is the thin Python binding."""
from . import build  # noqa: F401
