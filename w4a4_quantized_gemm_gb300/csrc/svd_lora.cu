// LoRA correction of the INT4 weights from W alone ("W4A4 CUDA Kernel for
// Voice Clone", 2.1: the quantisation error E = W - Q(W) is approximated by
// its rank-r SVD, L_up = (U_r S_r)^T, L_down = V_r; 2.2: rounds that quantise
// W - LoRA_previous and refit the SVD to the new error, stopping once the
// error no longer falls), with the round-to-nearest quantiser of the packer in
// place of GPTQ (no calibration data).
//
// The rank-r SVD is a randomized subspace iteration (Halko, Martinsson and
// Tropp, "Finding structure with randomness", 2011, Algorithm 4.4) on a block
// of s = 64 or 128 columns: Y = A Omega; q times { Z = orth(A^T Q); Q = orth(A Z) };
// B^T = A^T Q; the eigen-decomposition B B^T = W diag(lambda) W^T gives
// U = Q W, S = sqrt(lambda), V = B^T W / S.  Orthonormalisation is shifted
// Cholesky QR applied twice (Fukaya, Kannan, Nakatsukasa, Yamamoto and Yanagisawa,
// "Shifted Cholesky QR for computing the QR factorization of ill-conditioned
// matrices", 2020): G = Y^T Y (fp64), G + s I = R^T R with s = 1e-11 tr(G),
// Y <- Y R^-1; the shift keeps the factorisation defined for the rank-deficient
// blocks of an exactly low-rank error, the second pass restores orthogonality.
// The final eigen-decomposition is cyclic Jacobi (parallel round-robin order)
// in fp64 in one CTA, where eigenvalues below 1e-10 of the largest (singular
// values below 1e-5, fp32 rounding noise) are dropped.  The residual
// ||E - U S V^T||_F^2 = ||E||_F^2 - sum_{i<r} lambda_i.
//
// All arithmetic runs in these kernels; the host only sequences the launches
// and reads each round's error (the rounds stop on it).
#include <vector>

#include "kernels.h"

namespace w4a4 {
namespace {

constexpr int kRowsPerCta = 32;  // rows of A (nn) or columns of A (tn) per CTA of the thin products
constexpr int kChunk = 32;       // inner dimension per shared-memory stage

// Counter-based uniform numbers in [-1, 1): splitmix64 (Steele, Lea and Flood,
// "Fast splittable pseudorandom number generators", 2014) of (seed, index).
__global__ void fill_uniform_kernel(float* __restrict__ out, long long n, unsigned long long seed) {
    const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= n) return;
    unsigned long long z = seed + 0x9E3779B97F4A7C15ull * (unsigned long long)(i + 1);
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    z ^= z >> 31;
    out[i] = float((z >> 40) * (1.0 / 16777216.0)) * 2.0f - 1.0f;
}

// C[L, S] = A[L, Kd] . X[Kd, S]  (row-major, Kd % 32 == 0), fp32.
// CTA: 32 rows of A and all S columns; thread: one column quad, S/32 rows.
template <int S>
__global__ void __launch_bounds__(256) thin_nn_kernel(const float* __restrict__ A, int L, int Kd, int lda,
                                                      const float* __restrict__ X, int ldx,
                                                      float* __restrict__ C, int ldc) {
    constexpr int Q4 = S / 4, RG = 256 / Q4, RPT = kRowsPerCta / RG;
    static_assert(256 % Q4 == 0 && kRowsPerCta % RG == 0, "thread map must tile the 32 x S block");
    __shared__ float as[kRowsPerCta][kChunk + 1];
    __shared__ __align__(16) float xs[kChunk][S];
    const int t = threadIdx.x, cq = t % Q4, rg = t / Q4;
    const int row0 = blockIdx.x * kRowsPerCta;
    float acc[RPT][4] = {};
    for (int k0 = 0; k0 < Kd; k0 += kChunk) {
        for (int e = t; e < kRowsPerCta * kChunk; e += 256) {
            const int rr = e / kChunk, kk = e % kChunk;
            as[rr][kk] = row0 + rr < L ? A[(size_t)(row0 + rr) * lda + k0 + kk] : 0.f;
        }
        for (int e = t; e < kChunk * Q4; e += 256) {
            const int kk = e / Q4, c4 = e % Q4;
            *reinterpret_cast<float4*>(&xs[kk][4 * c4]) =
                *reinterpret_cast<const float4*>(X + (size_t)(k0 + kk) * ldx + 4 * c4);
        }
        __syncthreads();
#pragma unroll 8
        for (int kk = 0; kk < kChunk; ++kk) {
            const float4 xv = *reinterpret_cast<const float4*>(&xs[kk][4 * cq]);
#pragma unroll
            for (int i = 0; i < RPT; ++i) {
                const float a = as[rg + i * RG][kk];
                acc[i][0] = fmaf(a, xv.x, acc[i][0]);
                acc[i][1] = fmaf(a, xv.y, acc[i][1]);
                acc[i][2] = fmaf(a, xv.z, acc[i][2]);
                acc[i][3] = fmaf(a, xv.w, acc[i][3]);
            }
        }
        __syncthreads();
    }
#pragma unroll
    for (int i = 0; i < RPT; ++i) {
        const int rr = row0 + rg + i * RG;
        if (rr < L)
            *reinterpret_cast<float4*>(C + (size_t)rr * ldc + 4 * cq) =
                make_float4(acc[i][0], acc[i][1], acc[i][2], acc[i][3]);
    }
}

// C[Kd, S] = A[L, Kd]^T . Y[L, S], fp32.  CTA: 32 columns of A, all S columns
// of Y, the whole L in chunks of 32 rows.
template <int S>
__global__ void __launch_bounds__(256) thin_tn_kernel(const float* __restrict__ A, int L, int Kd, int lda,
                                                      const float* __restrict__ Y, int ldy,
                                                      float* __restrict__ C, int ldc) {
    constexpr int Q4 = S / 4, RG = 256 / Q4, RPT = kRowsPerCta / RG;
    static_assert(256 % Q4 == 0 && kRowsPerCta % RG == 0, "thread map must tile the 32 x S block");
    __shared__ float as[kChunk][kRowsPerCta + 1];  // [row of A][column of A]
    __shared__ __align__(16) float ys[kChunk][S];
    const int t = threadIdx.x, cq = t % Q4, rg = t / Q4;
    const int col0 = blockIdx.x * kRowsPerCta;
    float acc[RPT][4] = {};
    for (int n0 = 0; n0 < L; n0 += kChunk) {
        for (int e = t; e < kChunk * kRowsPerCta; e += 256) {
            const int nn = e / kRowsPerCta, cc = e % kRowsPerCta;
            as[nn][cc] = (n0 + nn < L && col0 + cc < Kd) ? A[(size_t)(n0 + nn) * lda + col0 + cc] : 0.f;
        }
        for (int e = t; e < kChunk * Q4; e += 256) {
            const int nn = e / Q4, c4 = e % Q4;
            *reinterpret_cast<float4*>(&ys[nn][4 * c4]) =
                n0 + nn < L ? *reinterpret_cast<const float4*>(Y + (size_t)(n0 + nn) * ldy + 4 * c4)
                            : make_float4(0.f, 0.f, 0.f, 0.f);
        }
        __syncthreads();
#pragma unroll 8
        for (int nn = 0; nn < kChunk; ++nn) {
            const float4 yv = *reinterpret_cast<const float4*>(&ys[nn][4 * cq]);
#pragma unroll
            for (int i = 0; i < RPT; ++i) {
                const float a = as[nn][rg + i * RG];
                acc[i][0] = fmaf(a, yv.x, acc[i][0]);
                acc[i][1] = fmaf(a, yv.y, acc[i][1]);
                acc[i][2] = fmaf(a, yv.z, acc[i][2]);
                acc[i][3] = fmaf(a, yv.w, acc[i][3]);
            }
        }
        __syncthreads();
    }
#pragma unroll
    for (int i = 0; i < RPT; ++i) {
        const int cc = col0 + rg + i * RG;
        if (cc < Kd)
            *reinterpret_cast<float4*>(C + (size_t)cc * ldc + 4 * cq) =
                make_float4(acc[i][0], acc[i][1], acc[i][2], acc[i][3]);
    }
}

// G[S, S] = M[L, S]^T M[L, S] in fp64; CTA (bi, bj) owns a 16 x 16 block.
__global__ void __launch_bounds__(256) gram_kernel(const float* __restrict__ M, int L, int S,
                                                   double* __restrict__ G) {
    __shared__ float mi[64][17], mj[64][17];
    const int ti = threadIdx.x / 16, tj = threadIdx.x % 16;
    const int bi = blockIdx.x * 16, bj = blockIdx.y * 16;
    double acc = 0.0;
    for (int n0 = 0; n0 < L; n0 += 64) {
        for (int e = threadIdx.x; e < 64 * 16; e += 256) {
            const int nn = e / 16, cc = e % 16;
            const bool ok = n0 + nn < L;
            mi[nn][cc] = ok ? M[(size_t)(n0 + nn) * S + bi + cc] : 0.f;
            mj[nn][cc] = ok ? M[(size_t)(n0 + nn) * S + bj + cc] : 0.f;
        }
        __syncthreads();
        for (int nn = 0; nn < 64; ++nn) acc += double(mi[nn][ti]) * double(mj[nn][tj]);
        __syncthreads();
    }
    G[(size_t)(bi + ti) * S + bj + tj] = acc;
}

// Eigen-decomposition of the symmetric S x S matrix G (fp64) by cyclic Jacobi
// sweeps in the parallel round-robin pair order (S/2 disjoint rotations per
// step, S - 1 steps per sweep), one CTA.  Writes eigenvalues lam[S] in
// descending order and the matching eigenvectors as columns of Wv[S][S].
// Also writes T = Wv diag(1 / sqrt(lam)) (directions with lam <= 1e-10 lam_max
// set to 0) when T is not null, and the sum of the first r eigenvalues.
__global__ void __launch_bounds__(1024) jacobi_eig_kernel(const double* __restrict__ G, int S, int r,
                                                          float* __restrict__ Wv, double* __restrict__ lam,
                                                          float* __restrict__ T, double* __restrict__ top_sum) {
    extern __shared__ double jm[];  // a[S][S] fp64, then v[S][S] fp32, pair table, rotations
    double* a = jm;
    float* v = reinterpret_cast<float*>(jm + S * S);
    int* pr = reinterpret_cast<int*>(v + S * S);  // pr[S]: round-robin positions
    double* cs = reinterpret_cast<double*>(pr + S + (S & 1));
    double* sn = cs + S / 2;
    int* ord = reinterpret_cast<int*>(sn + S / 2);
    __shared__ double off;
    const int tid = threadIdx.x, nt = blockDim.x;
    for (int e = tid; e < S * S; e += nt) {
        a[e] = G[e];
        v[e] = (e / S == e % S) ? 1.f : 0.f;
    }
    for (int e = tid; e < S; e += nt) pr[e] = e;
    __syncthreads();
    __shared__ double frob, red[32];
    auto block_sum = [&](double v) {  // fixed-order block reduction, result in red[0]
        for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
        __syncthreads();
        if ((tid & 31) == 0) red[tid >> 5] = v;
        __syncthreads();
        if (tid == 0) {
            double t = 0.0;
            for (int w = 0; w < (nt + 31) / 32; ++w) t += red[w];
            red[0] = t;
        }
        __syncthreads();
        return red[0];
    };
    {
        double f = 0.0;
        for (int e = tid; e < S * S; e += nt) f += a[e] * a[e];
        const double tf = block_sum(f);
        if (tid == 0) frob = tf;
    }
    __syncthreads();
    for (int sweep = 0; sweep < 30; ++sweep) {
        double o = 0.0;
        for (int e = tid; e < S * S; e += nt)
            if (e / S != e % S) o += a[e] * a[e];
        const double to = block_sum(o);
        if (tid == 0) off = to;
        __syncthreads();
        if (off <= 1e-28 * frob) break;
        for (int step = 0; step < S - 1; ++step) {
            // pairs (pr[i], pr[S-1-i]) for i < S/2: rotation angles
            for (int i = tid; i < S / 2; i += nt) {
                int p = pr[i], q = pr[S - 1 - i];
                if (p > q) { const int x = p; p = q; q = x; }
                const double apq = a[p * S + q], app = a[p * S + p], aqq = a[q * S + q];
                double c = 1.0, s = 0.0;
                if (fabs(apq) > 1e-300) {
                    const double th = (aqq - app) / (2.0 * apq);
                    const double tt = (th >= 0 ? 1.0 : -1.0) / (fabs(th) + sqrt(th * th + 1.0));
                    c = 1.0 / sqrt(tt * tt + 1.0);
                    s = tt * c;
                }
                cs[i] = c;
                sn[i] = s;
            }
            __syncthreads();
            // rows p, q of A (A <- J^T A)
            for (int e = tid; e < (S / 2) * S; e += nt) {
                const int i = e / S, j = e % S;
                int p = pr[i], q = pr[S - 1 - i];
                if (p > q) { const int x = p; p = q; q = x; }
                const double c = cs[i], s = sn[i];
                const double ap = a[p * S + j], aq = a[q * S + j];
                a[p * S + j] = c * ap - s * aq;
                a[q * S + j] = s * ap + c * aq;
            }
            __syncthreads();
            // columns p, q of A (A <- A J) and of V
            for (int e = tid; e < (S / 2) * S; e += nt) {
                const int i = e / S, j = e % S;
                int p = pr[i], q = pr[S - 1 - i];
                if (p > q) { const int x = p; p = q; q = x; }
                const double c = cs[i], s = sn[i];
                const double ap = a[j * S + p], aq = a[j * S + q];
                a[j * S + p] = c * ap - s * aq;
                a[j * S + q] = s * ap + c * aq;
                const float vp = v[j * S + p], vq = v[j * S + q];
                v[j * S + p] = float(c) * vp - float(s) * vq;
                v[j * S + q] = float(s) * vp + float(c) * vq;
            }
            __syncthreads();
            // next round-robin arrangement: position 0 fixed, the others rotate
            if (tid == 0) {
                const int last = pr[S - 1];
                for (int i = S - 1; i > 1; --i) pr[i] = pr[i - 1];
                pr[1] = last;
            }
            __syncthreads();
        }
    }
    // eigenvalues in descending order (selection by one thread; S <= 128)
    if (tid == 0) {
        for (int i = 0; i < S; ++i) ord[i] = i;
        for (int i = 0; i < S; ++i) {
            int best = i;
            for (int j = i + 1; j < S; ++j)
                if (a[ord[j] * S + ord[j]] > a[ord[best] * S + ord[best]]) best = j;
            const int x = ord[i]; ord[i] = ord[best]; ord[best] = x;
        }
        double ssum = 0.0;
        for (int i = 0; i < S; ++i) {
            lam[i] = a[ord[i] * S + ord[i]];
            if (i < r) ssum += lam[i] > 0.0 ? lam[i] : 0.0;
        }
        if (top_sum) *top_sum = ssum;
    }
    __syncthreads();
    const double lmax = a[ord[0] * S + ord[0]];
    for (int e = tid; e < S * S; e += nt) {
        const int row = e / S, col = e % S;
        const float w = v[row * S + ord[col]];
        Wv[e] = w;
        if (T) {
            const double l = a[ord[col] * S + ord[col]];
            T[e] = (l > 1e-10 * lmax && l > 0.0) ? float(double(w) / sqrt(l)) : 0.f;
        }
    }
}

// T = R^-1 (fp32, upper triangular) for G + s I = R^T R, s = 1e-11 tr(G), G
// fp64 S x S symmetric positive semidefinite; one CTA.  Right-looking
// Cholesky of the lower factor L = R^T in shared memory, then the columns of
// L^-1 by forward substitution, one column per thread; T = (L^-1)^T.
__global__ void __launch_bounds__(256) chol_inv_kernel(const double* __restrict__ G, int S,
                                                       float* __restrict__ T) {
    extern __shared__ double cm[];  // L [S][S] fp64, then X = L^-1 [S][S] fp32 (fp64 sums)
    double* a = cm;
    float* x = reinterpret_cast<float*>(cm + S * S);
    __shared__ double shift;
    const int tid = threadIdx.x, nt = blockDim.x;
    for (int e = tid; e < S * S; e += nt) a[e] = G[e];
    __syncthreads();
    if (tid == 0) {
        double tr = 0.0;
        for (int i = 0; i < S; ++i) tr += a[i * S + i];
        shift = tr > 0.0 ? 1e-11 * tr : 1e-300;
    }
    __syncthreads();
    for (int i = tid; i < S; i += nt) a[i * S + i] += shift;
    __syncthreads();
    for (int k = 0; k < S; ++k) {
        if (tid == 0) a[k * S + k] = sqrt(a[k * S + k] > shift ? a[k * S + k] : shift);
        __syncthreads();
        const double d = a[k * S + k];
        for (int i = k + 1 + tid; i < S; i += nt) a[i * S + k] /= d;
        __syncthreads();
        // trailing lower triangle: a[i][j] -= a[i][k] a[j][k], k < j <= i
        const int m = S - k - 1;
        for (int e = tid; e < m * m; e += nt) {
            const int i = k + 1 + e / m, j = k + 1 + e % m;
            if (j <= i) a[i * S + j] -= a[i * S + k] * a[j * S + k];
        }
        __syncthreads();
    }
    // X = L^-1, column c by forward substitution (threads over columns)
    for (int c = tid; c < S; c += nt) {
        for (int i = 0; i < S; ++i) {
            double v = (i == c) ? 1.0 : 0.0;
            for (int j = c; j < i; ++j) v -= a[i * S + j] * double(x[j * S + c]);
            x[i * S + c] = i < c ? 0.f : float(v / a[i * S + i]);
        }
    }
    __syncthreads();
    for (int e = tid; e < S * S; e += nt) {
        const int i = e / S, j = e % S;
        T[e] = x[j * S + i];  // (L^-1)^T: upper triangular R^-1
    }
}

// V[:, j] /= sqrt(lam[j]) for j < S (0 where lam_j <= 1e-10 lam_0); in place, V [K, S].
__global__ void scale_cols_kernel(float* __restrict__ V, long long K, int S, const double* __restrict__ lam) {
    const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= K * S) return;
    const int j = int(i % S);
    const double l = lam[j];
    V[i] = (l > 1e-10 * lam[0] && l > 0.0) ? float(double(V[i]) / sqrt(l)) : 0.f;
}

// Sum of squares of A [n elements] in fp64, one partial per CTA (fixed order).
__global__ void __launch_bounds__(256) sumsq_kernel(const float* __restrict__ A, long long n,
                                                    double* __restrict__ part) {
    __shared__ double red[256];
    double s = 0.0;
    for (long long i = (long long)blockIdx.x * 256 + threadIdx.x; i < n; i += (long long)gridDim.x * 256)
        s += double(A[i]) * double(A[i]);
    red[threadIdx.x] = s;
    __syncthreads();
    for (int o = 128; o > 0; o >>= 1) {
        if (threadIdx.x < o) red[threadIdx.x] += red[threadIdx.x + o];
        __syncthreads();
    }
    if (threadIdx.x == 0) part[blockIdx.x] = red[0];
}

// R[n, k] = W[n, k] - sum_{j < r} U[n, j] sig[j] V[k, j]  (U [N, ldu], V [K, ldv]).
__global__ void __launch_bounds__(256) residual_kernel(const float* __restrict__ W, int N, int K,
                                                       const float* __restrict__ U, int ldu,
                                                       const float* __restrict__ V, int ldv,
                                                       const double* __restrict__ lam, int r,
                                                       float* __restrict__ R) {
    __shared__ float us[32][129], vs[32][129];
    const int n0 = blockIdx.y * 32, k0 = blockIdx.x * 32;
    for (int e = threadIdx.x; e < 32 * r; e += 256) {
        const int i = e / r, j = e % r;
        const double l = lam[j];
        const float sg = l > 0.0 ? float(sqrt(l)) : 0.f;
        us[i][j] = n0 + i < N ? U[(size_t)(n0 + i) * ldu + j] * sg : 0.f;
        vs[i][j] = k0 + i < K ? V[(size_t)(k0 + i) * ldv + j] : 0.f;
    }
    __syncthreads();
    for (int e = threadIdx.x; e < 32 * 32; e += 256) {
        const int i = e / 32, kk = e % 32;
        if (n0 + i >= N || k0 + kk >= K) continue;
        float s = 0.f;
        for (int j = 0; j < r; ++j) s = fmaf(us[i][j], vs[kk][j], s);
        const size_t o = (size_t)(n0 + i) * K + k0 + kk;
        R[o] = W[o] - s;
    }
}

// E[n, k] = W[n, k] - code * fp16 scale, from the packed records.
__global__ void deq_error_kernel(const float* __restrict__ W, const uint8_t* __restrict__ packed, int N, int K,
                                 int r, float* __restrict__ E) {
    const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= (long long)N * K) return;
    const PackedLayout PL = packed_layout(N, K, r);
    const int n = int(i / K), k = int(i % K), g = k / kGroup, kk = k % kGroup;
    const int h = kk >> 5, k2 = kk & 31;
    const int q = (k2 & 15) >> 2, j = ((k2 >> 4) << 2) | (k2 & 3);
    const uint32_t word = reinterpret_cast<const uint32_t*>(packed + PL.qW)[((size_t)g * N + n) * 8 + 2 * q + h];
    const int code = int((word >> (4 * j)) & 15u) - 8;
    const float sc = __half2float(__ushort_as_half(reinterpret_cast<const uint16_t*>(packed + PL.sW)[(size_t)g * N + n]));
    E[i] = W[i] - float(code) * sc;
}

// L_down[k][j] = fp16(V[k][j]), L_up[j][n] = fp16(U[n][j] sqrt(lam[j])).
__global__ void lora_f16_kernel(const float* __restrict__ U, int N, const float* __restrict__ V, int K, int S,
                                const double* __restrict__ lam, int r, uint16_t* __restrict__ Ld,
                                uint16_t* __restrict__ Lu) {
    const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    if (i < (long long)K * r) {
        const int k = int(i / r), j = int(i % r);
        Ld[i] = __half_as_ushort(__float2half_rn(V[(size_t)k * S + j]));
    }
    if (i < (long long)r * N) {
        const int j = int(i / N), n = int(i % N);
        const double l = lam[j];
        const float sg = l > 0.0 ? float(sqrt(l)) : 0.f;
        Lu[i] = __half_as_ushort(__float2half_rn(U[(size_t)n * S + j] * sg));
    }
}

inline unsigned nblk(long long n, int per) { return unsigned((n + per - 1) / per); }

// block width of the subspace iteration for rank r: about min(3r, r + 64),
// rounded up to 64 or 128 (the widths the thin products are built for)
int block_cols(int r) {
    int s = 3 * r;
    if (s > r + 64) s = r + 64;
    return s <= 64 ? 64 : 128;
}

// Scratch carve-up (byte offsets, 256-aligned).
struct SvdScratch {
    size_t A, R, om, Y, Z, Bt, U, V, G, Wv, T, lam, sum, part, pk, total;
};
constexpr int kSumParts = 1024;
SvdScratch svd_scratch(int N, int K, int r) {
    const int S = block_cols(r);
    SvdScratch s{};
    size_t o = 0;
    auto take = [&](size_t bytes) { const size_t at = o; o = align256(o + bytes); return at; };
    s.A = take(sizeof(float) * size_t(N) * K);   // the matrix whose SVD is taken (the error E)
    s.R = take(sizeof(float) * size_t(N) * K);   // the residual W - LoRA handed to the quantiser
    s.om = take(sizeof(float) * size_t(K) * S);
    s.Y = take(sizeof(float) * size_t(N) * S);
    s.Z = take(sizeof(float) * size_t(K) * S);
    s.Bt = take(sizeof(float) * size_t(K) * S);
    s.U = take(sizeof(float) * size_t(N) * S);
    s.V = take(sizeof(float) * size_t(K) * S);
    s.G = take(sizeof(double) * S * S);
    s.Wv = take(sizeof(float) * S * S);
    s.T = take(sizeof(float) * S * S);
    s.lam = take(sizeof(double) * S);
    s.sum = take(sizeof(double) * 4);
    s.part = take(sizeof(double) * kSumParts);
    s.pk = take(packed_layout(N, K, r).total);  // the candidate round's packed weights
    s.total = o;
    return s;
}

struct Svd {
    int N, K, r, S;
    uint8_t* base;
    SvdScratch L;
    cudaStream_t st;
    float* f(size_t off) const { return reinterpret_cast<float*>(base + off); }
    double* d(size_t off) const { return reinterpret_cast<double*>(base + off); }

    template <int SS>
    void nn(const float* A, int rows, int inner, int lda, const float* X, float* C) const {
        thin_nn_kernel<SS><<<nblk(rows, kRowsPerCta), 256, 0, st>>>(A, rows, inner, lda, X, SS, C, SS);
    }
    template <int SS>
    void tn(const float* A, int rows, int cols, int lda, const float* Y, float* C) const {
        thin_tn_kernel<SS><<<nblk(cols, kRowsPerCta), 256, 0, st>>>(A, rows, cols, lda, Y, SS, C, SS);
    }
    size_t eig_smem() const {
        return sizeof(double) * S * S + sizeof(float) * S * S + sizeof(int) * (S + (S & 1)) +
               sizeof(double) * S + sizeof(int) * S;
    }
    // M [rows, S] <- M R^-1, twice (shifted Cholesky QR): orthonormal columns
    template <int SS>
    void orth(float* M, int rows, float* tmp) const {
        for (int pass = 0; pass < 2; ++pass) {
            gram_kernel<<<dim3(SS / 16, SS / 16), 256, 0, st>>>(M, rows, SS, d(L.G));
            chol_inv_kernel<<<1, 256, (sizeof(double) + sizeof(float)) * SS * SS, st>>>(d(L.G), SS, f(L.T));
            nn<SS>(M, rows, SS, SS, f(L.T), tmp);
            cudaMemcpyAsync(M, tmp, sizeof(float) * size_t(rows) * SS, cudaMemcpyDeviceToDevice, st);
        }
    }
    // rank-r SVD of the N x K matrix at L.A: U [N, S], V [K, S] (first r columns used),
    // eigenvalues lam[S] (singular values squared), sum of the first r at sum[0]
    template <int SS>
    void rsvd(int power, unsigned long long seed) const {
        const float* A = f(L.A);
        fill_uniform_kernel<<<nblk((long long)K * SS, 256), 256, 0, st>>>(f(L.om), (long long)K * SS, seed);
        nn<SS>(A, N, K, K, f(L.om), f(L.Y));
        orth<SS>(f(L.Y), N, f(L.U));
        for (int it = 0; it < power; ++it) {
            tn<SS>(A, N, K, K, f(L.Y), f(L.Z));
            orth<SS>(f(L.Z), K, f(L.V));
            nn<SS>(A, N, K, K, f(L.Z), f(L.Y));
            orth<SS>(f(L.Y), N, f(L.U));
        }
        tn<SS>(A, N, K, K, f(L.Y), f(L.Bt));                      // B^T = A^T Q
        gram_kernel<<<dim3(SS / 16, SS / 16), 256, 0, st>>>(f(L.Bt), K, SS, d(L.G));  // B B^T
        jacobi_eig_kernel<<<1, 1024, eig_smem(), st>>>(d(L.G), SS, r, f(L.Wv), d(L.lam), nullptr, d(L.sum));
        nn<SS>(f(L.Y), N, SS, SS, f(L.Wv), f(L.U));               // U = Q W
        nn<SS>(f(L.Bt), K, SS, SS, f(L.Wv), f(L.V));              // B^T W, then / sqrt(lam)
        scale_cols_kernel<<<nblk((long long)K * SS, 256), 256, 0, st>>>(f(L.V), K, SS, d(L.lam));
    }
    void rsvd_any(int power, unsigned long long seed) const {
        if (S == 64) rsvd<64>(power, seed);
        else rsvd<128>(power, seed);
    }
    // ||A||_F^2 in fp64 (the fixed-order sum of the per-CTA partials, on the host after a sync)
    double sumsq(const float* A, long long n) const {
        sumsq_kernel<<<kSumParts, 256, 0, st>>>(A, n, d(L.part));
        std::vector<double> h(kSumParts);
        cudaMemcpyAsync(h.data(), d(L.part), sizeof(double) * kSumParts, cudaMemcpyDeviceToHost, st);
        cudaStreamSynchronize(st);
        double s = 0.0;
        for (double x : h) s += x;
        return s;
    }
    double top_sum() const {
        double v = 0.0;
        cudaMemcpyAsync(&v, d(L.sum), sizeof(double), cudaMemcpyDeviceToHost, st);
        cudaStreamSynchronize(st);
        return v;
    }
};

w4a4_status eig_attr(int S) {
    const size_t smem = sizeof(double) * S * S + sizeof(float) * S * S + sizeof(int) * (S + (S & 1)) +
                        sizeof(double) * S + sizeof(int) * S;
    if (cudaFuncSetAttribute(jacobi_eig_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem)) !=
            cudaSuccess ||
        cudaFuncSetAttribute(chol_inv_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             int((sizeof(double) + sizeof(float)) * S * S)) != cudaSuccess)
        return W4A4_ERR_CUDA;
    return W4A4_OK;
}

}  // namespace

size_t svd_scratch_bytes(int N, int K, int r) { return svd_scratch(N, K, r).total; }

w4a4_status run_truncated_svd(const float* A, int N, int K, int r, int power, unsigned long long seed, float* U,
                              float* S_out, float* V, uint8_t* scratch, cudaStream_t st) {
    Svd s{N, K, r, block_cols(r), scratch, svd_scratch(N, K, r), st};
    w4a4_status e = eig_attr(s.S);
    if (e != W4A4_OK) return e;
    cudaMemcpyAsync(s.f(s.L.A), A, sizeof(float) * size_t(N) * K, cudaMemcpyDeviceToDevice, st);
    s.rsvd_any(power, seed);
    // first r columns of U, V and the singular values
    cudaMemcpy2DAsync(U, sizeof(float) * r, s.f(s.L.U), sizeof(float) * s.S, sizeof(float) * r, N,
                      cudaMemcpyDeviceToDevice, st);
    cudaMemcpy2DAsync(V, sizeof(float) * r, s.f(s.L.V), sizeof(float) * s.S, sizeof(float) * r, K,
                      cudaMemcpyDeviceToDevice, st);
    std::vector<double> lam(s.S);
    cudaMemcpyAsync(lam.data(), s.d(s.L.lam), sizeof(double) * s.S, cudaMemcpyDeviceToHost, st);
    if (cudaStreamSynchronize(st) != cudaSuccess) return W4A4_ERR_CUDA;
    std::vector<float> sg(r);
    for (int j = 0; j < r; ++j) sg[j] = lam[j] > 0.0 ? float(std::sqrt(lam[j])) : 0.f;
    cudaMemcpyAsync(S_out, sg.data(), sizeof(float) * r, cudaMemcpyHostToDevice, st);
    if (cudaStreamSynchronize(st) != cudaSuccess) return W4A4_ERR_CUDA;
    return launch_status();
}

w4a4_status run_svd_lora(const float* W, int N, int K, int r, int rounds, int power, unsigned long long seed,
                         uint8_t* packed, uint16_t* L_down, uint16_t* L_up, float* errs, uint8_t* scratch,
                         cudaStream_t st) {
    Svd s{N, K, r, block_cols(r), scratch, svd_scratch(N, K, r), st};
    w4a4_status e = eig_attr(s.S);
    if (e != W4A4_OK) return e;
    const long long nk = (long long)N * K;
    const size_t pk_bytes = packed_layout(N, K, r).total;
    double best = -1.0;
    for (int round = 0; round < rounds; ++round) {
        // quantise W - LoRA_previous (W itself in the first round) into the candidate buffer
        const float* Rin = W;
        if (round > 0) {
            residual_kernel<<<dim3(nblk(K, 32), nblk(N, 32)), 256, 0, st>>>(W, N, K, s.f(s.L.U), s.S, s.f(s.L.V),
                                                                            s.S, s.d(s.L.lam), r, s.f(s.L.R));
            Rin = s.f(s.L.R);
        }
        launch_pack_weights(Rin, nullptr, nullptr, N, K, r, 0, s.base + s.L.pk, st);
        // the error of this round's codes, and its rank-r SVD
        deq_error_kernel<<<nblk(nk, 256), 256, 0, st>>>(W, s.base + s.L.pk, N, K, r, s.f(s.L.A));
        const double e2 = s.sumsq(s.f(s.L.A), nk);
        s.rsvd_any(power, seed + 7919ull * (unsigned long long)round);
        const double top = s.top_sum();
        const double err = std::sqrt(e2 - top > 0.0 ? e2 - top : 0.0);
        if (errs) errs[round] = float(err);
        if (launch_status() != W4A4_OK) return W4A4_ERR_CUDA;
        if (best >= 0.0 && err >= best) {
            for (int k2 = round + 1; k2 < rounds; ++k2)
                if (errs) errs[k2] = -1.f;
            break;
        }
        best = err;
        // keep this round: its codes and scales, and its factors as fp16
        cudaMemcpyAsync(packed, s.base + s.L.pk, pk_bytes, cudaMemcpyDeviceToDevice, st);
        lora_f16_kernel<<<nblk((long long)(K > N ? K : N) * r, 256), 256, 0, st>>>(s.f(s.L.U), N, s.f(s.L.V), K, s.S,
                                                                                   s.d(s.L.lam), r, L_down, L_up);
        if (round + 1 == rounds)
            break;
    }
    launch_pack_lora(L_down, L_up, N, K, r, 0, packed, st);
    if (cudaStreamSynchronize(st) != cudaSuccess) return W4A4_ERR_CUDA;
    return launch_status();
}

}  // namespace w4a4
