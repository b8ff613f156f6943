// decode_splitkv_fp8.cu -- the split-KV decode over an e4m3 query and latent
// cache: decode_splitkv.cu compiled with MLA_F8 = 1 (mla_splitkv_kernel_f8).
#define MLA_F8 1
#include "decode_splitkv.cu"
