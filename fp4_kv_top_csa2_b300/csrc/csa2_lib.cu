// csa2_lib.cu -- the whole CSA2 CUDA library as one translation unit (one device module, so the
// kernels share the device status word and the compiler sees every call).
#include "kv_quant.cu"
#include "index_score.cu"
#include "index_mma.cu"
#include "index_multi.cu"
#include "topk.cu"
#include "attn_simt.cu"
#include "attn_mma.cu"
#include "attn_prefill.cu"
#include "attn_fp4pv.cu"
#include "index_keys.cu"
#include "api.cu"
#include "noalloc.cu"
