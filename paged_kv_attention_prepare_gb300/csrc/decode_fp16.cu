// The split-K kernel's fp16 instantiations (q, output and 16-bit pools in
// fp16), compiled apart from the bf16 ones in decode.cu so the two
// translation units build in parallel.  Everything else lives in decode.cu.
#define PA_DECODE_FP16_UNIT
#include "decode.cu"
