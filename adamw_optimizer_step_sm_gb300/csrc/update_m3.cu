// The update, one-launch device step and fused clipped step kernels of the
// bf16 without compensation (ADAMW_MODE_BF16_PLAIN) storage mode.
#define ADAMW_THIS_MODE 3
#include "update_mode.inc"
