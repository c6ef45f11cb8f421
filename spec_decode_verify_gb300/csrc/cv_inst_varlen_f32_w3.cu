// Packed-ragged-draft variants of the pipelined verify kernel for f32 elements, conv width 3 (units of at most 8 tokens).
#define CV_INST_VARLEN
#define CV_INST_B uint32_t
#define CV_INST_W 3
#define CV_INST_MAXT 8
#define CV_INST_NAME varlen_f32_w3
#include "cv_inst.cuh"
