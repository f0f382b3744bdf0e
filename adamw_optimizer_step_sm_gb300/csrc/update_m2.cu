// The update, one-launch device step and fused clipped step kernels of the
// mixed bf16 + remainder (ADAMW_MODE_MIXED_BF16_REMAINDER) storage mode.
#define ADAMW_THIS_MODE 2
#include "update_mode.inc"
