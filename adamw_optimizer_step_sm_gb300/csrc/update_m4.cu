// The update, one-launch device step and fused clipped step kernels of the
// bf16 Kahan with fp32 variance (ADAMW_MODE_BF16_KAHAN_FP32_VAR) storage mode.
#define ADAMW_THIS_MODE 4
#include "update_mode.inc"
