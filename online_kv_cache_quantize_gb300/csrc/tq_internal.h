// Internal declarations shared by the host set-up code and the CUDA sources
// of libtq. Not part of the public ABI (include/tq.h is).
#pragma once

#include <cstdint>
#include <string>
#include <vector>

#include "../../include/tq.h"

// two 32-bit words: the B-operand registers of one mma.sync fragment
struct uint2v {
    uint32_t x, y;
};

struct tq_rotation {
    int d = 0;
    int kind = 0;
    uint64_t seed = 0;
    std::vector<double> pi;     // d*d row-major, y = Pi x
    std::vector<double> signs;  // RHT sign layer (d), empty for dense
    int device = -1;            // device holding the copies, -1 = none
    float* d_pi32 = nullptr;    // Pi row-major fp32
    float* d_pit32 = nullptr;   // Pi^T row-major fp32 (PT[j][i] = Pi_ij)
    double* d_pi64 = nullptr;   // Pi row-major fp64 (exact re-decision path)
    float* d_sign = nullptr;    // RHT signs fp32 (d)
    uint2v* d_pi_frag = nullptr;  // d = 128 dense: 3 bf16 limbs of Pi^T in mma fragment order
    // d = 128: the tcgen05 quantize kernel's rotation operand W (y = W x / n,
    // scaled by 1/sqrt(d) for RHT) as bf16 128 x 128 tiles in the K-major
    // 128-byte-swizzled layout: 3 limbs of Pi (dense), H diag(s) (RHT, +-1)
    uint16_t* d_w_umma = nullptr;
};

struct tq_qjl {
    int m = 0;
    int d = 0;
    uint64_t seed = 0;
    std::vector<double> s;      // m*d row-major, bf16-exact values
    int device = -1;
    float* d_st32 = nullptr;    // S^T row-major fp32 (ST[i][j] = S_ji), [d][m]
    float* d_s32 = nullptr;     // S row-major fp32 [m][d]
    uint16_t* d_s16 = nullptr;  // m = d = 128: S as bf16 bits (exact), 16-byte unit (q, j) = S[j][8q .. 8q+7] at q * 128 + j
    uint2v* d_s_frag = nullptr;   // m = d = 128: S (exact bf16) in mma fragment order
    uint16_t* d_s_umma = nullptr; // m = d = 128: S as a bf16 tcgen05 operand (128-byte-swizzled layout)
};

namespace tq {

// host set-up math (host.cpp)
uint64_t splitmix64_at(uint64_t seed, uint64_t k);  // draw k (0-based)
void gaussians(uint64_t seed, int64_t count, double* out);
double round_bf16(double x);
void householder_haar(const double* g, int d, double* pi_out);  // Pi = Q diag(sign diag R)
tq_status codebook(int d, int bits, std::vector<double>& c, std::vector<double>& t);
// PolarQuant angle codebook of one level (1 = the coordinate pairs), ascending
tq_status polar_codebook(int level, int bits, std::vector<double>& c, std::vector<double>& t);

// thread-local error message
tq_status fail(tq_status s, const std::string& msg);
void clear_error();

// Bumped by every call that creates, uploads or frees a handle or flips a
// kernel switch: a prepared call is reused only while it is unchanged.
uint64_t handle_generation();
void bump_handle_generation();

}  // namespace tq
