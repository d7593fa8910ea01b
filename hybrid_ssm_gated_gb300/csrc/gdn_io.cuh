// gdn_io.cuh -- activation/output dtypes of a kernel instantiation.
//
// IO_ANY reads both dtypes from the launch arguments; every element load and
// store then branches on them. IO_BF16_F32 fixes bf16 activations and fp32
// outputs at compile time -- the common serving case -- so those branches fold
// away; the dispatchers pick it whenever the arguments match.
#pragma once

#include "gdn_device.cuh"

namespace gdn {

enum IoMode : int { IO_ANY = 0, IO_BF16_F32 = 1 };

template <int IO>
__device__ __forceinline__ int io_in(int runtime_dtype) {
    return IO == IO_BF16_F32 ? GDN_BF16 : runtime_dtype;
}

template <int IO>
__device__ __forceinline__ int io_out(int runtime_dtype) {
    return IO == IO_BF16_F32 ? GDN_F32 : runtime_dtype;
}

inline int io_mode(int in_dtype, int out_dtype) {
    return in_dtype == GDN_BF16 && out_dtype == GDN_F32 ? IO_BF16_F32 : IO_ANY;
}

}  // namespace gdn
