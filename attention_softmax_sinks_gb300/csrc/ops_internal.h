// Internal interface of the kernels around attention, as abi.cu sees it: the
// standalone router, QKV bias + rotary + K/V write, and the bias-seeded linear
// layer (each kernel file includes only its own header).
#pragma once
#include "linear_args.h"
#include "rope_args.h"
#include "router_args.h"
