// kq_inst_2.cu -- kernels for ntok = 2 (see kq_launch.cuh).
#include "kq_launch.cuh"

KQ_DEFINE_INSTANCES(2)
