// Host check of the piece schedule of the host-input step (fa_host_pieces in
// csrc/fa_internal.cuh, the function fa_constrained_step_host calls): for batches of
// 0 ... 20000 positions and a few large ones, the bounds start at 0, rise strictly, end at the
// batch size, number at most FA_HOST_PIECES (none for an empty batch), the first piece is a
// thirty-second of the batch (at least one position) and every piece but the last is at least
// the one before it and below 1.4 times one more than it (the sizes are the floors of a
// geometric series of ratio 1.4).  Prints "ok N" or the first failure.
#include <cstdio>

#include "../constrained_decoding_diffusion_gb300/csrc/fa_internal.cuh"

static bool check(size_t P) {
    size_t b[FA_HOST_PIECES + 1];
    const int n = fa_host_pieces(P, b);
    if (P == 0) return n == 0 && b[0] == 0;
    if (n < 1 || n > FA_HOST_PIECES || b[0] != 0 || b[n] != P) return false;
    for (int i = 0; i < n; ++i)
        if (b[i + 1] <= b[i]) return false;
    const size_t first = P / 32 > 0 ? P / 32 : 1;
    if (b[1] != (first < P ? first : P)) return false;
    for (int i = 1; i + 1 < n; ++i) {
        const double prev = (double)(b[i] - b[i - 1]), cur = (double)(b[i + 1] - b[i]);
        if (cur < prev || cur >= 1.4 * (prev + 1.0)) return false;
    }
    return true;
}

int main() {
    long checks = 0;
    for (size_t P = 0; P <= 20000; ++P, ++checks)
        if (!check(P)) { printf("bad pieces for P=%zu\n", P); return 1; }
    const size_t big[] = {8192, 65536, 1u << 20, 4294901760ull, 65535ull * 65536ull};
    for (size_t P : big) {
        ++checks;
        if (!check(P)) { printf("bad pieces for P=%zu\n", P); return 1; }
    }
    printf("ok %ld\n", checks);
    return 0;
}
