// The grouped (prefix-sharing) decode kernel, head_dim 64, reading its query
// and new rows with the lanes' copies (the mapped plan step).
#define PKV_D 64
#define PKV_G 8
#define PKV_GRP 1
#define PKV_MAPPED 1
#include "pkv_decode_inst.cuh"
