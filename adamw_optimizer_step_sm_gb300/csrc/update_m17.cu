// The update, one-launch device step and fused clipped step kernels of the
// any-precision storage mode ADAMW_MODE_ANYPREC | 1: bf16 param and grad,
// fp32 exp_avg, bf16 exp_avg_sq, bf16 compensation.
#define ADAMW_THIS_MODE (ADAMW_MODE_ANYPREC | 1)
#include "update_mode.inc"
