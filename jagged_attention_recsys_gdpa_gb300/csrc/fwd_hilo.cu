// The forward kernels for pointwise activations without the 1/Lkv normaliser
// (P enters the PV product as bf16 hi + lo parts); see the top of fwd.cu.
#define JATTN_HILO 1
#include "fwd.cu"
