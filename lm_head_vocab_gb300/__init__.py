"""lmloss for GB300: fused LM-head loss (collapse-free CE, z-loss, distillation
KL, GSPO) forward + backward over a [T, V] logit matrix, in hand-written
sm_103a CUDA behind a C ABI (include/lmloss.h)."""
from ._lib import LMLossError, build, load  # noqa: F401
from .lmloss import LMLoss, Outputs, lmloss_forward_backward  # noqa: F401
