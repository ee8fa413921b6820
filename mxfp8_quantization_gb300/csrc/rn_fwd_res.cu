// The row forward with a residual add (h = x + residual, stored, then
// normalized): the same kernel as rn_fwd.cu, instantiated with its RES flag
// set in a translation unit of its own so that the two halves compile in
// parallel.
#define RN_FWD_RES_TU 1
#include "rn_fwd.cu"
