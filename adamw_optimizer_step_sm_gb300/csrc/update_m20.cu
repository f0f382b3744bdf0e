// The update, one-launch device step and fused clipped step kernels of the
// any-precision storage mode ADAMW_MODE_ANYPREC | 4: bf16 param and grad,
// bf16 exp_avg, bf16 exp_avg_sq, fp32 compensation.
#define ADAMW_THIS_MODE (ADAMW_MODE_ANYPREC | 4)
#include "update_mode.inc"
