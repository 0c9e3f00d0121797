// Test shim: the Sequential Temperature Scaling root search of the CUDA
// library (sts_search.cuh), compiled for the host so that a CPU test can
// drive a whole fit with the same code the update kernel runs.
#include "sts_search.cuh"

extern "C" int sts_state_size() { return static_cast<int>(sizeof(dspark::StsState)); }
extern "C" int sts_search_step_host(dspark::StsState* s) { return dspark::sts_search_step(*s) ? 1 : 0; }
