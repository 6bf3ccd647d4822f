"""The bounds-checked build (-DMOE_CHECKED) compiles: every translation unit of
the library builds with the checks in (object files only, into a scratch
directory; the library itself is not replaced)."""
import concurrent.futures as cf
import importlib.util
import os
import subprocess

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _build_module():
    spec = importlib.util.spec_from_file_location("_moe_build", os.path.join(ROOT, "permute_grouped_expert_gb300",
                                                                            "_build.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def test_checked_build_compiles(tmp_path):
    b = _build_module()
    cc = b.nvcc()

    def compile_one(src):
        obj = os.path.join(str(tmp_path), os.path.basename(src) + ".o")
        r = subprocess.run([cc, *b.ARCH, *b.FLAGS, "-DMOE_CHECKED", "-c", src, "-o", obj], capture_output=True,
                           text=True)
        return src, r.returncode, r.stderr[-2000:]

    with cf.ThreadPoolExecutor(max_workers=min(8, os.cpu_count() or 4)) as ex:
        results = list(ex.map(compile_one, b._sources()))
    failed = [(os.path.basename(s), err) for s, rc, err in results if rc != 0]
    assert not failed, failed
