// Kernel instantiations for f32 keys.
#include "launch.cuh"

SEGTOPK_DEFINE_KEY_OPS(f32, segtopk::KeyKind::F32)
