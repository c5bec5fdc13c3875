// kq_inst_7.cu -- kernels for ntok = 7 (see kq_launch.cuh).
#include "kq_launch.cuh"

KQ_DEFINE_INSTANCES(7)
