// The update, one-launch device step and fused clipped step kernels of the
// mixed fp32 master (ADAMW_MODE_MIXED_FP32_MASTER) storage mode.
#define ADAMW_THIS_MODE 1
#include "update_mode.inc"
