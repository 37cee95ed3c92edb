// FlashAttention forward for FP32 inputs: the split pre-pass (each element as a bf16
// high part and a bf16 low part) and the 256-row prefill kernel of fa_prefill.cu built
// with its SPLIT option, which forms every product from the two parts. Compiled as a
// translation unit of its own so that the build compiles it beside fa_prefill.cu.
#define FA_PREFILL_SPLIT_TU 1
#include "fa_prefill.cu"
