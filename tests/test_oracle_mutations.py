"""The oracle's pins catch planted mistakes.

Each case copies the oracle's C source, plants one plausible mistake in the
copy (a dropped term or factor, a wrong sign, index, shift or byte order, a
transposed operand, another rounding), builds the copy as the oracle's
library in a child process, and runs the pin tests (test_oracle.py,
test_ptq1.py) against it there: the copy must build and at least one pin
must fail. The unmodified copy, built the same way, must pass them all.
The mistakes are planted in the oracle only, on the CPU.
"""
import os
import subprocess
import sys
import tempfile

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "tq_ref.c")
HDR = os.path.join(ROOT, "oracle", "tq_ref.h")

# (what the mistake is, text in tq_ref.c, the mistaken text)
MUTATIONS = [
    ("w = u + 1 instead of u - 1",
     "s += (pq2_code(blk, k) - 1) * q8K_value", "s += (pq2_code(blk, k) + 1) * q8K_value"),
    ("offset dropped: u * q instead of (u - 1) * q",
     "s += (pq2_code(blk, k) - 1) * q8K_value", "s += pq2_code(blk, k) * q8K_value"),
    ("activation of the mirrored column",
     "q8K_value(xq, nb, t, g * REF_GROUP + k);", "q8K_value(xq, nb, t, g * REF_GROUP + 127 - k);"),
    ("pq2_0 code byte k >> 3",
     "block[2 + (k >> 2)] >> (2 * (k & 3))", "block[2 + (k >> 3)] >> (2 * (k & 3))"),
    ("pq2_0 code shift k & 3 instead of 2 (k & 3)",
     "block[2 + (k >> 2)] >> (2 * (k & 3))", "block[2 + (k >> 2)] >> (k & 3)"),
    ("pq2_0 scale bytes swapped",
     "return (uint16_t)(block[0] | (block[1] << 8));", "return (uint16_t)(block[1] | (block[0] << 8));"),
    ("d_x of block g / 4 instead of g / 2",
     "const double dx = (double)xq[t * nb + g / 2].d;", "const double dx = (double)xq[t * nb + g / 4].d;"),
    ("d_w dropped",
     "const double term = dw * dx * isum;", "const double term = dx * isum;"),
    ("d_x dropped",
     "const double term = dw * dx * isum;", "const double term = dw * isum;"),
    ("rows of the output transposed with tokens",
     "y[t * rows + r] = (float)acc;", "y[r * ntok + t] = (float)acc;"),
    ("quantizer truncates instead of rounding",
     "long q = lrintf(p);", "long q = (long)p;"),
    ("quantizer rounds ties away from zero",
     "long q = lrintf(p);", "long q = lroundf(p);"),
    ("quantizer scale inverted",
     "yb->d = amax / 127.0f;", "yb->d = 127.0f / amax;"),
    ("quantizer scale from 128",
     "const float iscale = 127.0f / amax;", "const float iscale = 128.0f / amax;"),
    ("bsums over 8 values",
     "for (int j = 0; j < 16; ++j) s += yb->qs[16 * i + j];",
     "for (int j = 0; j < 8; ++j) s += yb->qs[16 * i + j];"),
    ("fp16 exponent bias off by one",
     "v = ldexpf((float)(1024 + m), e - 25);", "v = ldexpf((float)(1024 + m), e - 24);"),
    ("fp16 subnormal scale off by one",
     "v = ldexpf((float)m, -24);", "v = ldexpf((float)m, -25);"),
    ("tq layout: word and byte index transposed",
     "return (int64_t)h * 512 + l * 16 + wd * 4 + j;", "return (int64_t)h * 512 + l * 16 + j * 4 + wd;"),
    ("tq layout: slot shift from k % 4",
     "return 2 * ((k % 16) / 4);", "return 2 * (k % 4);"),
    ("tq layout: padding rows get code 0",
     "int u = 1;", "int u = 0;"),
    ("tq layout: scale bytes of the row swapped",
     "tile[TQ_CODE_BYTES + 2 * l] = (uint8_t)(sb & 0xFF);",
     "tile[TQ_CODE_BYTES + 2 * l] = (uint8_t)(sb >> 8);"),
    ("ptq1_0 trit divides by 255",
     "return (3 * v) / 256;", "return (3 * v) / 255;"),
    ("ptq1_0 byte rounds down",
     "return (uint8_t)((256 * q + 242) / 243);", "return (uint8_t)((256 * q) / 243);"),
    ("ptq1_0 trits in reverse order",
     "for (int n = 0; n < 5; ++n) q = 3 * q + t[n];", "for (int n = 0; n < 5; ++n) q = 3 * q + t[4 - n];"),
    ("ptq1_0 code byte k / 4",
     "const int u = ref_ptq1_trit(src[2 + k / 5], k % 5);",
     "const int u = ref_ptq1_trit(src[2 + k / 4], k % 5);"),
]

CHILD = r"""
import os, sys
root, tests, src, hdr, out = sys.argv[1:6]
sys.path[:0] = [root, tests]
import oracle
oracle._SRC, oracle._HDR, oracle._OUT_DIR = src, hdr, out
oracle._LIB = os.path.join(out, "libtq_ref.so")
oracle._lib = None
try:
    oracle.build()
except Exception as e:
    print("build failed:", e)
    sys.exit(10)
import pytest
sys.exit(pytest.main(["-x", "-q", "-p", "no:cacheprovider", "--rootdir", root,
                      os.path.join(tests, "test_oracle.py"), os.path.join(tests, "test_ptq1.py")]))
"""


def _run_pins(source_text):
    with tempfile.TemporaryDirectory() as d:
        src, hdr = os.path.join(d, "tq_ref.c"), os.path.join(d, "tq_ref.h")
        with open(src, "w") as f:
            f.write(source_text)
        with open(HDR) as f, open(hdr, "w") as g:
            g.write(f.read())
        p = subprocess.run([sys.executable, "-c", CHILD, ROOT, os.path.join(ROOT, "tests"), src,
                            hdr, d], capture_output=True, text=True, timeout=300, cwd=ROOT)
        return p.returncode, p.stdout + p.stderr


def _source():
    with open(SRC) as f:
        return f.read()


def test_unmodified_copy_passes_the_pins():
    rc, out = _run_pins(_source())
    assert rc == 0, out[-2000:]


@pytest.mark.parametrize("what,old,new", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_planted_mistake_fails_a_pin(what, old, new):
    src = _source()
    assert src.count(old) == 1, f"mutation site not unique: {old!r}"
    rc, out = _run_pins(src.replace(old, new))
    assert rc != 10, f"the mistaken copy did not build: {what}\n{out[-1500:]}"
    assert rc == 1, f"no pin caught: {what}\n{out[-1500:]}"
