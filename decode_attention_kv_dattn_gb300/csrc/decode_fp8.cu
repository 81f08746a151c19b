// The decode kernel over E4M3 (fp8) KV caches: the same source as decode.cu,
// instantiated with F8 = true in a translation unit of its own so that the
// two sets of kernels compile in parallel.
#define DATTN_DECODE_FP8_UNIT 1
#include "decode.cu"
