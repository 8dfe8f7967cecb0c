// Kernel instantiations for f16 keys.
#include "launch.cuh"

SEGTOPK_DEFINE_KEY_OPS(f16, segtopk::KeyKind::F16)
