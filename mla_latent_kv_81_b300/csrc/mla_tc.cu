// The tensor-core paths live in mla_decode_tc.cu (attention) and mla_gemm_tc.cu (projections).
#include "mla_tc.cuh"
