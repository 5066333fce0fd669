// The forward kernels for block masks: fwd.cu compiled with the block-mask
// arithmetic kept (see the top of fwd.cu).
#define JATTN_FWD_BLOCK 1
#include "fwd.cu"
