// Instantiations of the decode kernels for __nv_bfloat16 storage.
#include "decode_kernel.cuh"

namespace pkv {

const DecodeKernel* decode_kernel_bf16(int D, int B) {
    using dec::Launcher;
    switch (D * 1000 + B) {
        case 64008: return Launcher<__nv_bfloat16, 64, 8>::get();
        case 64016: return Launcher<__nv_bfloat16, 64, 16>::get();
        case 64032: return Launcher<__nv_bfloat16, 64, 32>::get();
        case 64064: return Launcher<__nv_bfloat16, 64, 64>::get();
        case 128008: return Launcher<__nv_bfloat16, 128, 8>::get();
        case 128016: return Launcher<__nv_bfloat16, 128, 16>::get();
        case 128032: return Launcher<__nv_bfloat16, 128, 32>::get();
        case 128064: return Launcher<__nv_bfloat16, 128, 64>::get();
        default: return nullptr;
    }
}

const DecodeKernel* decode_kernel_contig_bf16(int D) {
    using dec::Launcher;
    switch (D) {
        case 64: return Launcher<__nv_bfloat16, 64, step_tokens(64), kModeContig>::get();
        case 128: return Launcher<__nv_bfloat16, 128, step_tokens(128), kModeContig>::get();
        default: return nullptr;
    }
}

}  // namespace pkv
