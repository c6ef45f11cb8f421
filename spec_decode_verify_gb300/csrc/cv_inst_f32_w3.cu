// Kernel instantiations for f32 elements, conv width 3.
#define CV_INST_B uint32_t
#define CV_INST_W 3
#define CV_INST_MAXT 8
#define CV_INST_NAME kernels_f32_w3
#include "cv_inst.cuh"
