// Entry points whose kernels are not built yet: they validate nothing and
// report TS_ERR_UNSUPPORTED so callers fail loudly instead of silently.
#include "ts_common.cuh"

