// Kernel instantiations for f64 keys.
#include "launch.cuh"

SEGTOPK_DEFINE_KEY_OPS(f64, segtopk::KeyKind::F64)
