// Decode kernels for head_dim 64, 4 query head(s) per KV head.
#define PKV_D 64
#define PKV_G 4
#include "pkv_decode_inst.cuh"
