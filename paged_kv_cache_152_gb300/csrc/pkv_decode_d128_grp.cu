// The grouped (prefix-sharing) decode kernel, head_dim 128: 8 query rows per item.
#define PKV_D 128
#define PKV_G 8
#define PKV_GRP 1
#include "pkv_decode_inst.cuh"
