"""The boundary is a C ABI: include/fp4q.h compiles as plain C99 with
warnings as errors, and a C program links against libfp4q.so and calls it
(host-side paths only; no GPU needed)."""
import os
import subprocess

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_plain_c_client_builds_and_runs(tmp_path):
    from fp4_block_scaled_bf16_gb300 import build
    lib = build.build()
    exe = tmp_path / "abi_check"
    subprocess.run(["gcc", "-std=c99", "-Wall", "-Wextra", "-Werror", "-pedantic",
                    "-I", os.path.join(ROOT, "include"), os.path.join(ROOT, "tests", "abi_check.c"),
                    "-L", os.path.dirname(lib), "-lfp4q", "-Wl,-rpath," + os.path.dirname(lib),
                    "-o", str(exe)], check=True)
    r = subprocess.run([str(exe)], capture_output=True, text=True)
    assert r.returncode == 0 and r.stdout.strip() == "ok", r.stdout + r.stderr
