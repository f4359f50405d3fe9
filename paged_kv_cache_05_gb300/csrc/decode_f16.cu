// Instantiations of the decode kernels for __half storage.
#include "decode_kernel.cuh"

namespace pkv {

const DecodeKernel* decode_kernel_f16(int D, int B) {
    using dec::Launcher;
    switch (D * 1000 + B) {
        case 64008: return Launcher<__half, 64, 8>::get();
        case 64016: return Launcher<__half, 64, 16>::get();
        case 64032: return Launcher<__half, 64, 32>::get();
        case 64064: return Launcher<__half, 64, 64>::get();
        case 128008: return Launcher<__half, 128, 8>::get();
        case 128016: return Launcher<__half, 128, 16>::get();
        case 128032: return Launcher<__half, 128, 32>::get();
        case 128064: return Launcher<__half, 128, 64>::get();
        default: return nullptr;
    }
}

const DecodeKernel* decode_kernel_contig_f16(int D) {
    using dec::Launcher;
    switch (D) {
        case 64: return Launcher<__half, 64, step_tokens(64), kModeContig>::get();
        case 128: return Launcher<__half, 128, step_tokens(128), kModeContig>::get();
        default: return nullptr;
    }
}

}  // namespace pkv
