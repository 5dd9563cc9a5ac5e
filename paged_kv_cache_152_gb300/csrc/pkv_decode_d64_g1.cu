// Decode kernels for head_dim 64, 1 query head(s) per KV head.
#define PKV_D 64
#define PKV_G 1
#include "pkv_decode_inst.cuh"
