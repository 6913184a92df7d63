// Decode over FP8 pools with bf16 queries and outputs (the fp16 half and
// the dispatcher live in decode_fp8.cu).
#define PKV_FP8_IO_BF16
#include "decode_fp8.cu"
