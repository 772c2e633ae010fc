// Run-time compilation of a plan's tensor-product kernels for sm_103a (NVRTC),
// loaded through the CUDA runtime's context-independent library API.
#include <cuda_runtime.h>
#include <nvrtc.h>

#include <cstring>
#include <iterator>
#include <vector>
#include <string>

#include "internal.hpp"

namespace cgtp {

static const char* kKernelNames[] = {"cgtp_fwd_conv",   "cgtp_fwd_single",
                                     "cgtp_bwd_conv",   "cgtp_bwd_conv_nogy",
                                     "cgtp_bwd_single", "cgtp_bwd_single_nogy"};
static const char* kStagedNames[] = {"cgtp_fwd_conv_tma",   "cgtp_fwd_single_tma",
                                     "cgtp_bwd_conv_tma",   "cgtp_bwd_conv_nogy_tma",
                                     "cgtp_bwd_single_tma", "cgtp_bwd_single_nogy_tma"};

cgtp_status compile_module(const std::string& src, const std::string& name, Module& m,
                           std::string& err) {
    nvrtcProgram prog;
    if (nvrtcCreateProgram(&prog, src.c_str(), name.c_str(), 0, nullptr, nullptr) != NVRTC_SUCCESS) {
        err = "nvrtcCreateProgram failed";
        return CGTP_E_COMPILE;
    }
    const char* opts[] = {"-arch=sm_103a", "-std=c++17", "-lineinfo", "-DNDEBUG",
                          "--ptxas-options=-v"};
    nvrtcResult rc = nvrtcCompileProgram(prog, 5, opts);
    size_t logsz = 0;
    nvrtcGetProgramLogSize(prog, &logsz);
    std::string log(logsz, '\0');
    if (logsz) nvrtcGetProgramLog(prog, &log[0]);
    m.log = log;
    if (rc != NVRTC_SUCCESS) {
        err = std::string("NVRTC: ") + nvrtcGetErrorString(rc) + "\n" + log;
        nvrtcDestroyProgram(&prog);
        return CGTP_E_COMPILE;
    }
    size_t n = 0;
    nvrtcGetCUBINSize(prog, &n);
    m.cubin.resize(n);
    nvrtcGetCUBIN(prog, m.cubin.data());
    nvrtcDestroyProgram(&prog);
    return CGTP_OK;
}

cgtp_status load_module(Module& m, bool staged, std::string& err) {
    if (m.lib) return CGTP_OK;
    cudaLibrary_t lib = nullptr;
    cudaError_t ce = cudaLibraryLoadData(&lib, m.cubin.data(), nullptr, nullptr, 0, nullptr,
                                         nullptr, 0);
    if (ce != cudaSuccess) {
        set_cuda_error(ce);
        err = std::string("cudaLibraryLoadData: ") + cudaGetErrorString(ce);
        return CGTP_E_CUDA;
    }
    std::vector<const char*> names(std::begin(kKernelNames), std::end(kKernelNames));
    if (staged) names.insert(names.end(), std::begin(kStagedNames), std::end(kStagedNames));
    for (const char* k : names) {
        cudaKernel_t kern = nullptr;
        ce = cudaLibraryGetKernel(&kern, lib, k);
        if (ce != cudaSuccess) {
            set_cuda_error(ce);
            err = std::string("cudaLibraryGetKernel(") + k + "): " + cudaGetErrorString(ce);
            cudaLibraryUnload(lib);
            return CGTP_E_CUDA;
        }
        m.kernels[k] = kern;
    }
    m.lib = lib;
    if (cudaLibraryGetGlobal(&m.err_flag, nullptr, lib, "cgtp_device_error") != cudaSuccess) {
        m.err_flag = nullptr;
        cudaGetLastError();
    }
    return CGTP_OK;
}

Module::~Module() {
    if (lib) cudaLibraryUnload(lib);
}

// The plan's module: compiled once (host only), loaded on first GPU use.
cgtp_status get_module(Plan& p, bool load, std::shared_ptr<Module>& out, std::string& err) {
    std::lock_guard<std::mutex> g(p.mu);
    auto it = p.modules.find("tp");
    std::shared_ptr<Module> m;
    if (it == p.modules.end()) {
        m = std::make_shared<Module>();
        cgtp_status st = compile_module(p.kernel_source(), "cgtp_tp.cu", *m, err);
        if (st != CGTP_OK) return st;
        p.modules["tp"] = m;
    } else {
        m = it->second;
    }
    if (load) {
        cgtp_status st = load_module(*m, p.staged, err);
        if (st != CGTP_OK) return st;
    }
    out = m;
    return CGTP_OK;
}

}  // namespace cgtp
