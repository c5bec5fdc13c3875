// kq_inst_8.cu -- kernels for ntok = 8 (see kq_launch.cuh).
#include "kq_launch.cuh"

KQ_DEFINE_INSTANCES(8)
