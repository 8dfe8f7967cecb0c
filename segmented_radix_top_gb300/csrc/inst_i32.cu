// Kernel instantiations for i32 keys.
#include "launch.cuh"

SEGTOPK_DEFINE_KEY_OPS(i32, segtopk::KeyKind::I32)
