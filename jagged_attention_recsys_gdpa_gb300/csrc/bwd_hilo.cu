// The backward kernels for pointwise activations without the 1/Lkv
// normaliser (P and dS enter the second products as bf16 hi + lo parts); see
// the top of bwd.cu.
#define JATTN_HILO 1
#include "bwd.cu"
