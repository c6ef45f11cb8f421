// Packed-ragged-draft variants of the pipelined verify kernel for bf16 elements, conv width 3 (units of at most 8 tokens).
#define CV_INST_VARLEN
#define CV_INST_B uint16_t
#define CV_INST_W 3
#define CV_INST_MAXT 8
#define CV_INST_NAME varlen_bf16_w3
#include "cv_inst.cuh"
