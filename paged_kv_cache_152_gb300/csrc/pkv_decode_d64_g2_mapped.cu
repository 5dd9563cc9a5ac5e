// Decode kernels for head_dim 64, 2 query head(s) per KV head, reading their
// query and new rows with the lanes' copies (the mapped plan step).
#define PKV_D 64
#define PKV_G 2
#define PKV_MAPPED 1
#include "pkv_decode_inst.cuh"
