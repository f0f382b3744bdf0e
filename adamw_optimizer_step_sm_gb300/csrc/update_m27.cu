// The update, one-launch device step and fused clipped step kernels of the
// any-precision storage mode ADAMW_MODE_ANYPREC | 11: bf16 param and grad,
// fp32 exp_avg, fp32 exp_avg_sq, no compensation.
#define ADAMW_THIS_MODE (ADAMW_MODE_ANYPREC | 11)
#include "update_mode.inc"
