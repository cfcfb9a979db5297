// The backward's kernels and C entry points (attn_bwd.cu) built for the host:
// see emu_device.h in this directory. Compiled by tests/test_backward_emulated.py.
#define SSA_HOST_EMULATION 1
#include "attn_bwd.cu"
