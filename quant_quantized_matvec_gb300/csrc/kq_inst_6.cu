// kq_inst_6.cu -- kernels for ntok = 6 (see kq_launch.cuh).
#include "kq_launch.cuh"

KQ_DEFINE_INSTANCES(6)
