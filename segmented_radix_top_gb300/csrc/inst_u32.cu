// Kernel instantiations for u32 keys.
#include "launch.cuh"

SEGTOPK_DEFINE_KEY_OPS(u32, segtopk::KeyKind::U32)
