// Instantiations of the decode kernels that write each sequence's newest
// token (kModeAppend) for __half storage.
#include "decode_kernel.cuh"

namespace pkv {

const DecodeKernel* decode_kernel_append_f16(int D, int B) {
    using dec::Launcher;
    switch (D * 1000 + B) {
        case 64008: return Launcher<__half, 64, 8, kModeAppend>::get();
        case 64016: return Launcher<__half, 64, 16, kModeAppend>::get();
        case 64032: return Launcher<__half, 64, 32, kModeAppend>::get();
        case 64064: return Launcher<__half, 64, 64, kModeAppend>::get();
        case 128008: return Launcher<__half, 128, 8, kModeAppend>::get();
        case 128016: return Launcher<__half, 128, 16, kModeAppend>::get();
        case 128032: return Launcher<__half, 128, 32, kModeAppend>::get();
        case 128064: return Launcher<__half, 128, 64, kModeAppend>::get();
        default: return nullptr;
    }
}

}  // namespace pkv
