// The block-mask forward kernels for pointwise activations without the 1/Lkv
// normaliser (P enters the PV product as bf16 hi + lo parts); see fwd.cu.
#define JATTN_FWD_BLOCK 1
#define JATTN_HILO 1
#include "fwd.cu"
