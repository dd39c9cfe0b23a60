// s5_backward_tc.cu -- the backward scan of the bidirectional layer
// ("Simplified State Space Layers for Sequence Modeling", "Paper vs code": a
// forward and a backward scan, C~ with 2P columns): the tensor-core kernel of
// s5_forward_tc.cu compiled with S5_TC_REV = 1 (chunks and tokens visited in
// reverse, the readout added into y).  A separate translation unit keeps the
// forward kernel's code exactly as it is without the backward variant.
#define S5_TC_REV 1
#include "s5_forward_tc.cu"
