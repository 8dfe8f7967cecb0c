// Kernel instantiations for bf16 keys.
#include "launch.cuh"

SEGTOPK_DEFINE_KEY_OPS(bf16, segtopk::KeyKind::BF16)
