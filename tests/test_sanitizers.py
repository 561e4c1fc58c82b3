"""Host code under AddressSanitizer and UndefinedBehaviorSanitizer, on the CPU.

compute-sanitizer is not available on the GPU pool, so the host side is
checked here instead: the CPU oracle, and the library's argument checking,
workspace carving and one-call paths (api.cu, noalloc.cu, host_pipe.cu,
and SageBwd's sagebwd.cu),
built with -fsanitize=address,undefined and driven by the two C programs in
tests/sanitize/ through every path that needs no device.  Any memory error or
undefined behaviour aborts the program, and the test fails.
"""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SAN = ["-fsanitize=address,undefined", "-fno-sanitize-recover=all", "-fno-omit-frame-pointer", "-g"]
ENV = dict(os.environ, ASAN_OPTIONS="detect_leaks=0:abort_on_error=1", UBSAN_OPTIONS="print_stacktrace=1",
           OMP_NUM_THREADS="4")


def _have_sanitizers():
    out = subprocess.run(["gcc", "-print-file-name=libasan.so"], capture_output=True, text=True).stdout.strip()
    return os.path.isabs(out) and os.path.exists(out)


pytestmark = pytest.mark.skipif(not _have_sanitizers(), reason="gcc without the sanitizer runtimes")


def _run(cmd, **kw):
    r = subprocess.run(cmd, capture_output=True, text=True, **kw)
    assert r.returncode == 0, f"{' '.join(cmd[:3])} ...\n{r.stdout[-3000:]}\n{r.stderr[-6000:]}"
    return r


def test_oracle_under_sanitizers(tmp_path):
    exe = tmp_path / "oracle_driver"
    _run(["gcc", "-O1", "-std=c11", "-fopenmp", "-ffp-contract=off", *SAN, "-I", os.path.join(ROOT, "oracle"),
          os.path.join(ROOT, "oracle", "sage_oracle.c"), os.path.join(ROOT, "oracle", "sagebwd_oracle.c"),
          os.path.join(ROOT, "tests", "sanitize", "oracle_driver.c"),
          "-o", str(exe), "-lm"])
    r = _run([str(exe)], env=ENV, timeout=600)
    assert "oracle driver: ok" in r.stdout


def test_abi_argument_checks_under_sanitizers(tmp_path):
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(nvcc):
        pytest.skip("nvcc not found")
    from bit_attention_gb300 import build
    build.build()  # the kernel objects come from the regular build
    csrc = os.path.join(ROOT, "bit_attention_gb300", "csrc")
    flags = build.ARCH + ["-O1", "-std=c++17", "-Xcompiler", "-fPIC", "--expt-relaxed-constexpr",
                          "-I", os.path.join(ROOT, "include")]
    # nvcc splits -Xcompiler values at commas: one flag per sanitizer
    for s in ["-fsanitize=address", "-fsanitize=undefined", "-fno-sanitize-recover=all",
              "-fno-omit-frame-pointer", "-g"]:
        flags += ["-Xcompiler", s]
    procs, objs = [], []
    for name in ("api", "noalloc", "host_pipe", "sagebwd"):
        obj = tmp_path / f"{name}.o"
        objs.append(str(obj))
        procs.append(subprocess.Popen([nvcc, *flags, "-c", os.path.join(csrc, name + ".cu"), "-o", str(obj)],
                                      stdout=subprocess.PIPE, stderr=subprocess.PIPE, text=True))
    for p in procs:
        out, err = p.communicate(timeout=900)
        assert p.returncode == 0, err[-4000:]
    kernels = [os.path.join(build.OUT, f"{n}.o") for n in ("attn", "quant", "probe")]
    lib = tmp_path / "libsagefp4_san.so"
    _run([nvcc, *build.ARCH, "-shared", "-o", str(lib), *objs, *kernels])
    exe = tmp_path / "abi_driver"
    _run(["gcc", "-O1", "-std=c11", *SAN, "-I", os.path.join(ROOT, "include"),
          os.path.join(ROOT, "tests", "sanitize", "abi_driver.c"), "-o", str(exe), "-L", str(tmp_path),
          "-lsagefp4_san", f"-Wl,-rpath,{tmp_path}"])
    r = _run([str(exe)], env=ENV, timeout=300)
    assert "abi driver: ok" in r.stdout
