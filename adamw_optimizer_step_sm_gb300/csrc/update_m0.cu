// The update, one-launch device step and fused clipped step kernels of the
// bf16 Kahan (ADAMW_MODE_BF16_KAHAN) storage mode.
#define ADAMW_THIS_MODE 0
#include "update_mode.inc"
