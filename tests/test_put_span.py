"""Byte shuffles of the vector path and the ring, compiled on the host from
the shipped source text of csrc/snac.cuh: the store at another 16-byte
phase (put_span, put_span_words) and the fixed-offset window of the ragged
ring's shifted copies (window_at).

A ReduceScatter(V) window on the sources' grid ends at an arbitrary
destination phase: put_span stores bytes [b0, b0 + nb) of a 16-byte sum at
an address aligned only to the element size.  The functions are cut out of
the header, compiled with g++ against stand-ins for the device intrinsics
they use (a 128-bit store, a byte shift of a vector pair, a funnel shift,
make_uint4), and run for every destination phase, first byte and length:
exactly the window's bytes must change, to the right values, and every
store must be naturally aligned and inside the window.  window_at must
return bytes [4K + r/8, 4K + r/8 + 16) of its 32-byte pair for every word
offset K and bit shift r.  Planted mistakes in the cut-out text must be
caught.
"""
import os
import re
import shutil
import subprocess

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))
SNAC = os.path.join(os.path.dirname(HERE), "collective_datapath_atom_gb300", "csrc", "snac.cuh")

PRELUDE = r"""
#include <cstdint>
#include <cstdio>
#include <cstring>
struct uint4 { uint32_t x, y, z, w; };
static uint4 make_uint4(uint32_t x, uint32_t y, uint32_t z, uint32_t w) { return uint4{x, y, z, w}; }
static int bad = 0;
static uint8_t *lo_, *hi_;
static void check(const char *p, int size) {
    if ((uintptr_t)p % size) { std::printf("misaligned %d-byte store\n", size); bad = 1; }
    if ((const uint8_t *)p < lo_ || (const uint8_t *)p + size > hi_) {
        std::printf("store outside the window\n");
        bad = 1;
    }
}
namespace atom {
static void st_v4(char *d, uint4 v) { check(d, 16); std::memcpy(d, &v, 16); }
static uint4 shift_pair(uint4 a, uint4 b, uint32_t sh) {
    uint8_t t[32];
    std::memcpy(t, &a, 16);
    std::memcpy(t + 16, &b, 16);
    uint4 r;
    std::memcpy(&r, t + sh, 16);
    return r;
}
}  // namespace atom
static uint32_t __funnelshift_r(uint32_t lo, uint32_t hi, uint32_t s) {
    return (uint32_t)((((uint64_t)hi << 32) | lo) >> (s & 31));
}
template <class T> struct Ref {
    char *p;
    void operator=(T v) { check(p, sizeof(T)); std::memcpy(p, &v, sizeof(T)); }
};
template <class T> struct Ptr {
    char *p;
    Ref<T> operator*() { return Ref<T>{p}; }
};
template <class PT> struct Cast;
template <class T> struct Cast<T *> { static Ptr<T> of(char *p) { return Ptr<T>{p}; } };
template <class PT> static auto store_cast(char *p) { return Cast<PT>::of(p); }
"""

MAIN = r"""
template <int ES> static void run() {
    for (uint32_t ph = 0; ph < 16; ph += ES)
        for (uint32_t b0 = 0; b0 < 16; b0 += ES)
            for (uint32_t nb = ES; b0 + nb <= 16; nb += ES) {
                alignas(16) uint8_t buf[64];
                std::memset(buf, 0xEE, sizeof buf);
                uint8_t src[16];
                for (int i = 0; i < 16; ++i) src[i] = (uint8_t)(i * 17 + 3);
                uint4 v;
                std::memcpy(&v, src, 16);
                char *d = (char *)buf + 16 + ph;
                lo_ = (uint8_t *)d;
                hi_ = (uint8_t *)d + nb;
                put_span<ES>(d, v, b0, nb);
                for (int i = 0; i < 64; ++i) {
                    const int rel = i - 16 - (int)ph;
                    const uint8_t want = rel >= 0 && rel < (int)nb ? src[b0 + rel] : 0xEE;
                    if (buf[i] != want) {
                        std::printf("ES=%d phase=%u b0=%u nb=%u: byte %d\n", ES, ph, b0, nb, rel);
                        bad = 1;
                        return;
                    }
                }
            }
}
int main() {
    run<2>();
    run<4>();
    std::printf(bad ? "FAIL\n" : "ok\n");
    return bad;
}
"""


def cut_functions():
    """put_span_words and put_span, as they stand in the header."""
    text = open(SNAC).read()
    start = text.index("template <int ES>\n__device__ __forceinline__ void put_span_words(")
    end = text.index("// One 16-byte window of a segment")
    body = text[start:end].replace("__device__ __forceinline__", "static inline")
    body = re.sub(r"reinterpret_cast<(uint32_t|uint16_t) \*>\(", r"store_cast<\1 *>(", body)
    assert "put_span(" in body and "__device__" not in body
    return body


@pytest.fixture(scope="module")
def compile_and_run(tmp_path_factory):
    gxx = shutil.which("g++")
    if gxx is None:
        pytest.skip("no host C++ compiler")
    d = tmp_path_factory.mktemp("put_span")

    def go(body, name):
        src = d / f"{name}.cpp"
        src.write_text(PRELUDE + body + MAIN)
        exe = d / name
        subprocess.run([gxx, "-std=c++17", "-O1", str(src), "-o", str(exe)], check=True)
        return subprocess.run([str(exe)], capture_output=True, text=True)

    return go


def test_put_span_stores_exactly_the_window(compile_and_run):
    res = compile_and_run(cut_functions(), "shipped")
    assert res.returncode == 0, res.stdout


@pytest.mark.parametrize("plant", [
    # a word straddling the source words read from the wrong end
    ("__funnelshift_r(w[i], w[i + 1], 16)", "__funnelshift_r(w[i + 1], w[i], 16)"),
    # the last half word of a 2-mod-4 destination dropped
    ("if ((nb - 2) & 2u)", "if (false)"),
])
def test_the_harness_catches_a_planted_mistake(compile_and_run, plant):
    body = cut_functions()
    assert plant[0] in body
    res = compile_and_run(body.replace(plant[0], plant[1]), "planted")
    assert res.returncode != 0 and "FAIL" in res.stdout


WINDOW_MAIN = r"""
template <int K> static void check_k() {
    uint8_t pair[32];
    for (int i = 0; i < 32; ++i) pair[i] = (uint8_t)(i * 29 + 7);
    uint4 a, b;
    std::memcpy(&a, pair, 16);
    std::memcpy(&b, pair + 16, 16);
    for (uint32_t r = 0; r < 32; r += 8) {
        const uint4 w = window_at<K>(a, b, r);
        uint8_t got[16];
        std::memcpy(got, &w, 16);
        const uint32_t sh = 4 * K + r / 8;   // the window starts at byte sh of the pair
        for (int i = 0; i < 16; ++i)
            if (got[i] != pair[sh + i]) {
                std::printf("K=%d r=%u: byte %d\n", K, r, i);
                bad = 1;
                return;
            }
    }
}
int main() {
    check_k<0>();
    check_k<1>();
    check_k<2>();
    check_k<3>();
    std::printf(bad ? "FAIL\n" : "ok\n");
    return bad;
}
"""


def cut_window():
    text = open(SNAC).read()
    start = text.index("template <int K>\n__device__ __forceinline__ uint4 window_at(")
    end = text.index("\n}\n", start) + 3
    body = text[start:end].replace("__device__ __forceinline__", "static inline")
    assert "window_at(" in body and "__device__" not in body
    return body


def test_window_at_is_the_byte_window_of_the_pair(tmp_path):
    gxx = shutil.which("g++")
    if gxx is None:
        pytest.skip("no host C++ compiler")
    for name, body in (("shipped", cut_window()),
                       ("planted", cut_window().replace("w[K + 3], w[K + 4], r)",
                                                        "w[K + 3], w[K + 3], r)"))):
        src = tmp_path / f"{name}.cpp"
        src.write_text(PRELUDE + body + WINDOW_MAIN)
        exe = tmp_path / name
        subprocess.run([gxx, "-std=c++17", "-O1", str(src), "-o", str(exe)], check=True)
        res = subprocess.run([str(exe)], capture_output=True, text=True)
        if name == "shipped":
            assert res.returncode == 0, res.stdout
        else:
            assert res.returncode != 0 and "FAIL" in res.stdout
