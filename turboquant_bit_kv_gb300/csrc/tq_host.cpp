// Host-only parts of libtq: Lloyd-Max codebooks, sign diagonal, sizes and
// status strings.  No CUDA here.
//
// Codebook: "TurboQuant KV Cache Compression — Spec", Algorithm Detail Step 2
// and Codebook Generation.  The coordinate law of a rotated, L2-normalised
// vector is taken as y = 2u - 1 with u ~ Beta(d/2, d/2), whose density in y is
// proportional to (1 - y^2)^(d/2 - 1).  Lloyd's iteration alternates
// "boundary = midpoint of adjacent centroids" and "centroid = conditional mean
// of its cell"; the conditional means are ratios of integrals of y w(y) and
// w(y) over the cell, so the normalising constant of the law cancels.  The
// integrals use composite Gauss-Legendre quadrature (16 nodes per panel of
// width at most 1/128) on [-0.75, 0.75]; outside that interval w(y) is below
// 1e-22 of its peak for d = 128, far under double precision of the cell
// integrals.  The iteration starts from evenly spaced levels within +-2.5
// standard deviations (every cell has mass) and stops when no centroid moves
// by 1e-15; centroids are kept exactly antisymmetric, so the middle boundary
// is exactly 0.
//
// Signs: splitmix64 (Steele, Lea, Flood 2014), output j gives sign j.

#include "tq.h"

#include <cmath>
#include <cstring>
#include <mutex>

namespace {

constexpr int kD = 128;

struct GaussLegendre16 {
    double x[16], w[16];
    GaussLegendre16() {
        // Newton's method on P_16 from the Chebyshev-like initial guesses;
        // weights 2 / ((1 - x^2) P'(x)^2).
        const int n = 16;
        for (int i = 0; i < n; ++i) {
            double z = std::cos(M_PI * (i + 0.75) / (n + 0.5));
            double dp = 0.0;
            for (int it = 0; it < 100; ++it) {
                double p0 = 1.0, p1 = z;
                for (int k = 1; k < n; ++k) {
                    double p2 = ((2.0 * k + 1.0) * z * p1 - k * p0) / (k + 1.0);
                    p0 = p1;
                    p1 = p2;
                }
                dp = n * (z * p1 - p0) / (z * z - 1.0);
                double dz = p1 / dp;
                z -= dz;
                if (std::fabs(dz) < 1e-17) break;
            }
            x[i] = z;
            w[i] = 2.0 / ((1.0 - z * z) * dp * dp);
        }
    }
};

const GaussLegendre16 &gl16() {
    static const GaussLegendre16 g;
    return g;
}

// Integrals of w(y) and y w(y) over [a, b], w(y) = (1 - y^2)^(alpha - 1).
void cell_integrals(double a, double b, double alpha, double *m0, double *m1) {
    const double lim = 0.75;
    if (a < -lim) a = -lim;
    if (b > lim) b = lim;
    *m0 = 0.0;
    *m1 = 0.0;
    if (b <= a) return;
    const GaussLegendre16 &g = gl16();
    int panels = (int)std::ceil((b - a) * 128.0);
    if (panels < 1) panels = 1;
    double h = (b - a) / panels;
    double s0 = 0.0, s1 = 0.0;
    for (int p = 0; p < panels; ++p) {
        double lo = a + p * h, mid = lo + 0.5 * h;
        for (int i = 0; i < 16; ++i) {
            double y = mid + 0.5 * h * g.x[i];
            double wy = std::exp((alpha - 1.0) * std::log1p(-y * y)) * g.w[i];
            s0 += wy;
            s1 += y * wy;
        }
    }
    *m0 = 0.5 * h * s0;
    *m1 = 0.5 * h * s1;
}

void lloyd_beta(int d, int bits, double *c, double *b) {
    const int L = 1 << bits;
    const double alpha = d / 2.0;
    const double sigma = 1.0 / std::sqrt(d + 1.0);
    for (int i = 0; i < L; ++i) c[i] = 2.5 * sigma * (2.0 * (i + 0.5) / L - 1.0);
    double nc[16];
    for (int it = 0; it < 200000; ++it) {
        for (int i = 0; i + 1 < L; ++i) b[i] = 0.5 * (c[i] + c[i + 1]);
        for (int i = 0; i < L; ++i) {
            double lo = (i == 0) ? -1.0 : b[i - 1];
            double hi = (i == L - 1) ? 1.0 : b[i];
            double m0, m1;
            cell_integrals(lo, hi, alpha, &m0, &m1);
            nc[i] = m1 / m0;
        }
        double delta = 0.0;
        for (int i = 0; i < L; ++i) {
            double v = 0.5 * (nc[i] - nc[L - 1 - i]);
            delta = std::fmax(delta, std::fabs(v - c[i]));
            c[i] = v;
        }
        if (delta < 1e-15) break;
    }
    for (int i = 0; i + 1 < L; ++i) b[i] = 0.5 * (c[i] + c[i + 1]);
}

std::mutex g_cb_mutex;
// cached codebooks per (head dim 64 / 96 / 128 / 160, bits)
constexpr int kCbDims[4] = {64, 96, 128, 160};
bool g_cb_ready[4][5] = {};
tq_codebook g_cb[4][5];

}  // namespace

extern "C" int tq_codebook_load(int head_dim, int bits, tq_codebook *out) {
    if (!out) return TQ_ERR_ARG;
    if (head_dim == kD && bits == 8) {
        // turboq8: the uniform grid (i - 127.5) / 127.5 is implicit; no table
        std::memset(out, 0, sizeof(*out));
        out->head_dim = head_dim;
        out->bits = 8;
        out->levels = 256;
        return TQ_OK;
    }
    int di = -1;
    for (int i = 0; i < 4; ++i)
        if (kCbDims[i] == head_dim) di = i;
    if (di < 0 || bits < 2 || bits > 4) return TQ_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_cb_mutex);
    if (!g_cb_ready[di][bits]) {
        double c[16] = {0}, b[15] = {0};
        lloyd_beta(head_dim, bits, c, b);
        tq_codebook cb;
        std::memset(&cb, 0, sizeof(cb));
        cb.head_dim = head_dim;
        cb.bits = bits;
        cb.levels = 1 << bits;
        for (int i = 0; i < cb.levels; ++i) cb.centroids[i] = (float)c[i];
        for (int i = 0; i + 1 < cb.levels; ++i) cb.boundaries[i] = (float)b[i];
        g_cb[di][bits] = cb;
        g_cb_ready[di][bits] = true;
    }
    *out = g_cb[di][bits];
    return TQ_OK;
}

extern "C" int tq_signs_from_seed(uint64_t seed, int head_dim, tq_signs *out) {
    if (!out) return TQ_ERR_ARG;
    if (head_dim != kD) return TQ_ERR_UNSUPPORTED;
    std::memset(out, 0, sizeof(*out));
    uint64_t state = seed;
    for (int j = 0; j < kD; ++j) {
        state += 0x9E3779B97F4A7C15ull;
        uint64_t z = state;
        z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
        z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
        z ^= z >> 31;
        if (z >> 63) out->w[j >> 5] |= 1u << (j & 31);
    }
    return TQ_OK;
}

extern "C" size_t tq_block_bytes(int bits) {
    if (bits == 8) return 130;
    if (bits < 2 || bits > 4) return 0;
    return 2 + (size_t)kD * bits / 8;
}

extern "C" size_t tq_serde_size(int num_layers, int num_tokens, int hidden_dim, int head_dim,
                                int block_size, int skip_first, int skip_last,
                                int key_bits, int value_bits, int elem_bytes) {
    if (num_layers < 0 || num_tokens < 0 || hidden_dim <= 0 || head_dim != kD ||
        hidden_dim % head_dim || block_size <= 0 || skip_first < 0 || skip_last < 0 ||
        tq_block_bytes(key_bits) == 0 || tq_block_bytes(value_bits) == 0 || elem_bytes != 2)
        return 0;
    int qs = skip_first < num_layers ? skip_first : num_layers;
    int qe = num_layers - skip_last;
    if (qe < qs) qe = qs;
    size_t heads = (size_t)(hidden_dim / head_dim);
    size_t nblk = ((size_t)num_tokens + block_size - 1) / block_size;
    size_t slot = tq_block_bytes(key_bits) + tq_block_bytes(value_bits);
    size_t raw_layers = (size_t)(num_layers - (qe - qs));
    return 2 * raw_layers * (size_t)num_tokens * hidden_dim * elem_bytes +
           (size_t)(qe - qs) * nblk * block_size * heads * slot;
}

extern "C" const char *tq_status_string(int status) {
    switch (status) {
        case TQ_OK: return "ok";
        case TQ_ERR_ARG: return "invalid argument";
        case TQ_ERR_UNSUPPORTED: return "unsupported head_dim, bits, dtype or group size";
        case TQ_ERR_ALIGN: return "misaligned pointer or stride";
        case TQ_ERR_WORKSPACE: return "workspace too small";
        case TQ_ERR_CUDA: return "CUDA error";
        case TQ_ERR_TIMEOUT: return "a kernel gave up a bounded wait (its output is invalid)";
        default: return "unknown status";
    }
}
