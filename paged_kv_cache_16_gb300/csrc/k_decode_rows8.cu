// The split-KV decode kernels specialised for launches whose items all have
// at most 8 (query token, head) rows -- every decode row with G <= 8: MMA rows
// 8..15 are padding, so their q fragments and accumulators are dropped.
#define PA_DECODE_ROWS8 1
#include "k_decode.cu"
