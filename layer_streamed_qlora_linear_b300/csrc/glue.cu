// placeholder, filled in with the stack glue kernels
#include "common.cuh"
