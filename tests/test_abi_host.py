"""Host-side checks of the C ABI (no GPU needed): exports, validation, planning logic."""
import os
import re

import pytest
import torch

from dense_gemm_hgemm_gb300 import workloads

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HAS_GPU = torch.cuda.is_available()


def _declared_functions():
    names = set()
    for h in os.listdir(os.path.join(ROOT, "include")):
        text = open(os.path.join(ROOT, "include", h), encoding="utf-8").read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        names |= set(re.findall(r"\b((?:gemm|tma)_[a-z_0-9]+)\s*\(", text))
    return sorted(names)


def test_header_declares_the_boundary():
    names = _declared_functions()
    for required in ("gemm_plan_create", "gemm_run", "gemm_plan_destroy", "gemm_plan_check",
                     "gemm_status_string"):
        assert required in names


def test_library_exports_every_declared_symbol(gemm_lib):
    lib = gemm_lib.library()
    missing = [n for n in _declared_functions() if not hasattr(lib, n)]
    assert not missing, missing


def test_exported_symbols_are_c_linkage(gemm_lib):
    import subprocess
    out = subprocess.run(["nm", "-D", "--defined-only", gemm_lib.LIB_PATH] if hasattr(gemm_lib, "LIB_PATH")
                         else ["nm", "-D", "--defined-only", gemm_lib._build.LIB_PATH],
                         capture_output=True, text=True, check=True).stdout
    exported = set(line.split()[-1] for line in out.splitlines() if line.strip())
    for n in _declared_functions():
        assert n in exported, n


def test_abi_version_and_status_strings(gemm_lib):
    assert gemm_lib.gemm_abi_version() == 1
    for code, name in gemm_lib.STATUS_NAMES.items():
        assert gemm_lib.gemm_status_string(code).startswith(name)
    assert "unknown" in gemm_lib.gemm_status_string(1234)


def _create_status(g, M, N, K, dtype, layout=0):
    import ctypes
    h = ctypes.c_void_p()
    st = g.library().gemm_plan_create(M, N, K, dtype, layout, ctypes.byref(h))
    if st == 0:
        g.gemm_plan_destroy(h.value)
    return st


@pytest.mark.parametrize("args,expect", [
    ((64, 64, 64, 7, 0), 2),        # unknown dtype
    ((64, 64, 64, 0, 4), 2),        # unknown layout
    ((60, 64, 64, 0, 2), 3),        # A stored K x M: M*2 bytes not a multiple of 16
    ((64, 60, 64, 0, 1), 3),        # B stored K x N: N*2 bytes not a multiple of 16
    ((64, 64, 60, 0, 3), 0 if HAS_GPU else 4),   # NT: K is never a stored row; passes validation
    ((-1, 64, 64, 0, 0), 1),        # negative M
    ((64, -8, 64, 0, 0), 1),
    ((64, 64, -8, 1, 0), 1),
    ((64, 64, 60, 0, 0), 3),        # K*2 bytes not a multiple of 16
    ((64, 60, 64, 0, 0), 3),        # N*2 bytes not a multiple of 16
    ((64, 64, 40, 2, 0), 3),        # int8: K must be a multiple of 16
    ((64, 62, 64, 2, 0), 3),        # int32 C: N must be a multiple of 4
    ((2 ** 31, 64, 64, 0, 0), 1),   # beyond 32-bit indices
])
def test_create_validates_before_touching_the_device(gemm_lib, args, expect):
    assert _create_status(gemm_lib, *args) == expect


@pytest.mark.skipif(HAS_GPU, reason="checks the no-device path")
def test_create_without_gpu_reports_no_device(gemm_lib):
    assert _create_status(gemm_lib, 128, 128, 64, 0) == 4


def test_vectorcall_entry_points_match_ctypes(gemm_lib):
    """The CPython entry points of gemm_run / gemm_launch_empty are built with the
    library and return what the ctypes calls return (no device needed)."""
    import dense_gemm_hgemm_gb300 as g
    lib = g.library()                                         # loads both
    pc = g._pycall
    assert pc is not None, "_gemm_pycall was not built"
    assert pc.run(0, 0, 0, 0, 0) == lib.gemm_run(None, None, None, None, None) == 1
    assert pc.run(0, 16, 32, 48, 0) == 1                      # null plan: invalid argument
    with pytest.raises(TypeError):
        pc.run(0, 0, 0)
    with pytest.raises(TypeError):
        pc.run(0, "A", 0, 0, 0)                                 # not an address
    with pytest.raises(g.GemmError) as e:
        g.gemm_run(0, None, None, None, 0)
    assert e.value.status == 1


def test_null_handles(gemm_lib):
    lib = gemm_lib.library()
    assert lib.gemm_plan_destroy(None) == 0
    assert lib.gemm_run(None, None, None, None, None) == 1
    assert lib.gemm_plan_check(None, None) == 1
    assert lib.gemm_plan_get_config(None, None) == 1
    assert lib.gemm_plan_get_launch(None, None, None, None) == 1
    assert lib.gemm_plan_set_timeout(None, 5) == 1
    assert lib.gemm_plan_create(64, 64, 64, 0, 0, None) == 1


def test_select_config_valid_for_every_workload(gemm_lib):
    shapes = [(w.M, w.N, w.K, w.dtype) for w in workloads.NAMED + tuple(workloads.sweep_shapes())]
    for M, N, K, dt in shapes:
        c = gemm_lib.gemm_select_config(M, N, K, dt, 152)
        bn = c["block_n"]
        assert bn in (64, 128, 224, 256), (M, N, K, c)
        assert bn != 224 or (c["cta_pair"] == 1 and c["split_k"] == 1), (M, N, K, c)
        if dt == "i8" and bn > 128:   # wide integer tiles: SM pairs, one K slice
            assert c["cta_pair"] == 1 and c["split_k"] == 1 and c["multicast"] == 0, (M, N, K, c)
        assert c["stages"] in (3, 4, 6, 8)
        num_kb = -(-K // 64)
        assert 1 <= c["split_k"] <= num_kb
        per = -(-num_kb // c["split_k"])
        assert (c["split_k"] - 1) * per < num_kb          # no empty K slice
        assert 1 <= c["raster_group"]


def test_select_config_big_shapes_fill_the_gpu(gemm_lib):
    for w in (workloads.SQUARE_8192, workloads.FFN_BF16, workloads.INT8_4096):
        c = gemm_lib.gemm_select_config(w.M, w.N, w.K, w.dtype, 152)
        tiles = -(-w.M // 128) * -(-w.N // c["block_n"])
        assert tiles >= 152 and c["split_k"] == 1


def test_cost_model_matches_the_tables_sm_pair_choice(gemm_lib):
    """Off the table (M shifted by 8 rows, the same tile counts) the cost model
    chooses SM pairs exactly where the measured table does."""
    import json
    from dense_gemm_hgemm_gb300 import tune
    doc = json.load(open(tune.TUNED_JSON))
    n = 0
    for r in doc["shapes"]:
        if r["dtype"] != "f16" or r["M"] < 256:
            continue
        c = gemm_lib.gemm_select_config(r["M"] - 8, r["N"], r["K"], "f16", 152)
        assert c["cta_pair"] == r["best"]["cta_pair"], (r, c)
        n += 1
    assert n > 200


def test_cost_model_configs_are_valid_off_the_table(gemm_lib):
    """Seeded random shapes (mostly off the table): the chosen configuration is one
    that plan validation accepts."""
    import random
    rnd = random.Random(11)
    for _ in range(600):
        dt = rnd.choice(("f16", "bf16", "i8"))
        M = rnd.randint(1, 12000)
        N = rnd.randint(1, 3000) * 4 if dt == "i8" else rnd.randint(1, 1500) * 8
        K = rnd.randint(1, 800) * (16 if dt == "i8" else 8)
        c = gemm_lib.gemm_select_config(M, N, K, dt, 152)
        assert gemm_lib.gemm_workspace_bytes(M, N, K, dt, c) >= 0, (M, N, K, dt, c)


def test_select_config_splits_k_for_few_tiles(gemm_lib):
    c = gemm_lib.gemm_select_config(128, 128, 4096, "f16", 152)
    assert c["split_k"] > 1


def test_cluster_split_validation(gemm_lib):
    ok = gemm_lib.gemm_workspace_bytes(128, 128, 4096, "f16",
                                       {"block_n": 64, "split_k": 4, "split_mode": 1})
    base = gemm_lib.gemm_workspace_bytes(128, 128, 4096, "f16", {"block_n": 64, "split_k": 1})
    assert ok == base                      # cluster split needs no plan scratch
    for bad in ({"block_n": 64, "split_k": 3, "split_mode": 1},      # 128 rows / 3
                {"block_n": 64, "split_k": 16, "split_mode": 1},     # beyond a portable cluster
                {"block_n": 64, "split_k": 2, "split_mode": 7}):
        with pytest.raises(gemm_lib.GemmError):
            gemm_lib.gemm_workspace_bytes(128, 128, 4096, "f16", bad)


@pytest.mark.parametrize("mb,nb,g", [(1, 1, 1), (7, 3, 2), (64, 32, 16), (33, 57, 8), (5, 9, 16)])
def test_raster_is_a_bijection(gemm_lib, mb, nb, g):
    seen = set()
    for t in range(mb * nb):
        m, n = gemm_lib.gemm_tile_coords(mb, nb, g, t)
        assert 0 <= m < mb and 0 <= n < nb
        seen.add((m, n))
    assert len(seen) == mb * nb


def test_raster_bands_keep_concurrent_tiles_compact(gemm_lib):
    # 152 consecutive tiles of a 64 x 32 grid in bands of 16 m-blocks touch at
    # most 16 m-blocks and ceil(152/16)+1 n-blocks.
    ms, ns = set(), set()
    for t in range(152):
        m, n = gemm_lib.gemm_tile_coords(64, 32, 16, t)
        ms.add(m)
        ns.add(n)
    assert len(ms) <= 16 and len(ns) <= 11


def test_workspace_bytes(gemm_lib):
    base = gemm_lib.gemm_workspace_bytes(128, 128, 4096, "f16", {"block_n": 128, "split_k": 1})
    split = gemm_lib.gemm_workspace_bytes(128, 128, 4096, "f16", {"block_n": 128, "split_k": 4})
    assert split - base >= 4 * 128 * 128 * 4
    i8 = gemm_lib.gemm_workspace_bytes(256, 512, 1024, "i8", {"block_n": 128})
    assert i8 >= (256 + 512) * 1024 * 2
    with pytest.raises(gemm_lib.GemmError):
        gemm_lib.gemm_workspace_bytes(128, 128, 64, "i8", {"block_n": 256})
    with pytest.raises(gemm_lib.GemmError):
        gemm_lib.gemm_workspace_bytes(128, 128, 64, "f16", {"block_n": 96})
    with pytest.raises(gemm_lib.GemmError):
        gemm_lib.gemm_workspace_bytes(128, 128, 64, "f16", {"block_n": 128, "stages": 3})


def test_product_path_has_no_oracle_or_fallback():
    """The package never imports the oracle, torch matmul or another GEMM backend."""
    pkg = os.path.join(ROOT, "dense_gemm_hgemm_gb300")
    banned = re.compile(r"import oracle|from oracle|torch\.matmul|cublas|triton|np\.dot|\.mm\(|einsum|bmm")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h", ".inc")):
                text = open(os.path.join(dirpath, f), encoding="utf-8").read()
                assert not banned.search(text), (f, banned.search(text).group(0))


def test_config_table_is_the_emitted_sweep(tmp_path):
    """csrc/gemm_config_table.inc is exactly what tune.py emits from tuned_configs.json."""
    from dense_gemm_hgemm_gb300 import tune
    out = tmp_path / "table.inc"
    tune.emit(tune.TUNED_JSON, str(out))
    assert out.read_text() == open(tune.TABLE).read()


def test_table_covers_the_sweep_and_named_shapes(gemm_lib):
    import json
    from dense_gemm_hgemm_gb300 import tune
    doc = json.load(open(tune.TUNED_JSON))
    have = {(r["M"], r["N"], r["K"], r["dtype"]) for r in doc["shapes"]}
    for w in list(workloads.sweep_shapes()) + list(workloads.NAMED):
        assert (w.M, w.N, w.K, w.dtype) in have
    for r in doc["shapes"]:
        c = gemm_lib.gemm_select_config(r["M"], r["N"], r["K"], r["dtype"], 152)
        for k, v in r["best"].items():
            assert c[k] == v or (k == "raster_group" and c[k] <= v), (r, c)


def test_pair_config_validation(gemm_lib):
    ok = gemm_lib.gemm_workspace_bytes(4096, 4096, 4096, "f16", {"block_n": 256, "cta_pair": 1})
    assert ok > 0
    base = gemm_lib.gemm_workspace_bytes(1024, 1024, 4096, "f16", {"block_n": 256, "cta_pair": 1})
    for s in (2, 4):   # K slices across the pairs of one cluster of 2 * s CTAs: no scratch
        cfg = {"block_n": 256, "cta_pair": 1, "split_k": s, "split_mode": 1}
        assert gemm_lib.gemm_workspace_bytes(1024, 1024, 4096, "f16", cfg) == base
    for dtype, bad in (("i8", {"block_n": 256, "cta_pair": 1, "split_k": 2, "split_mode": 1}),
                       ("f16", {"block_n": 64, "cta_pair": 1}),
                       ("f16", {"block_n": 256, "cta_pair": 1, "split_k": 2}),
                       ("f16", {"block_n": 256, "cta_pair": 1, "split_k": 8, "split_mode": 1}),
                       ("f16", {"block_n": 256, "cta_pair": 1, "stages": 4}),
                       ("f16", {"block_n": 256, "cta_pair": 3})):
        with pytest.raises(gemm_lib.GemmError):
            gemm_lib.gemm_workspace_bytes(4096, 4096, 4096, dtype, bad)


def test_pair_224_config_validation(gemm_lib):
    """224-wide tiles: SM pairs, one K slice, no multicast."""
    for dtype in ("f16", "bf16", "i8"):
        for ks in (1, 2):
            cfg = {"block_n": 224, "cta_pair": 1, "kblocks_per_stage": ks}
            assert gemm_lib.gemm_workspace_bytes(4096, 4096, 4096, dtype, cfg) > 0
    for dtype, bad in (("f16", {"block_n": 224}),
                       ("f16", {"block_n": 224, "cta_pair": 1, "split_k": 2, "split_mode": 1}),
                       ("f16", {"block_n": 224, "cta_pair": 1, "split_k": 2}),
                       ("f16", {"block_n": 224, "cta_pair": 1, "multicast": 2}),
                       ("f16", {"block_n": 224, "cta_pair": 1, "stages": 8}),
                       ("f16", {"block_n": 224, "cta_pair": 1, "kblocks_per_stage": 4}),
                       ("i8", {"block_n": 224})):
        with pytest.raises(gemm_lib.GemmError):
            gemm_lib.gemm_workspace_bytes(4096, 4096, 4096, dtype, bad)


def test_wide_integer_tile_validation(gemm_lib):
    """int8 -> int32 wider than 128 columns: SM pairs only, one K slice, no multicast."""
    for bn in (224, 256):
        for ks in (1, 2):
            cfg = {"block_n": bn, "cta_pair": 1, "kblocks_per_stage": ks}
            assert gemm_lib.gemm_workspace_bytes(1024, 1024, 4096, "i8", cfg) > 0
        for bad in ({"block_n": bn},
                    {"block_n": bn, "cta_pair": 1, "split_k": 2, "split_mode": 1},
                    {"block_n": bn, "cta_pair": 1, "multicast": 2}):
            with pytest.raises(gemm_lib.GemmError):
                gemm_lib.gemm_workspace_bytes(1024, 1024, 4096, "i8", bad)


def test_multicast_config_validation(gemm_lib):
    ok = gemm_lib.gemm_workspace_bytes(1024, 1024, 4096, "f16", {"block_n": 64, "multicast": 4})
    assert ok == gemm_lib.gemm_workspace_bytes(1024, 1024, 4096, "f16", {"block_n": 64})
    for bad in ({"block_n": 64, "multicast": 3},
                {"block_n": 64, "multicast": 8},
                {"block_n": 64, "multicast": 2, "split_k": 2},
                {"block_n": 256, "multicast": 4, "cta_pair": 1},
                {"block_n": 256, "multicast": 2, "cta_pair": 1, "split_k": 2, "split_mode": 1},
                {"block_n": 128, "multicast": 2, "cta_pair": 1, "kblocks_per_stage": 2}):
        with pytest.raises(gemm_lib.GemmError):
            gemm_lib.gemm_workspace_bytes(1024, 1024, 4096, "f16", bad)
    # two SM pairs sharing A (a four-CTA cluster)
    for cfg in ({"block_n": 256, "multicast": 2, "cta_pair": 1},
                {"block_n": 128, "multicast": 2, "cta_pair": 1}):
        assert gemm_lib.gemm_workspace_bytes(1024, 1024, 4096, "f16", cfg) > 0


def test_multicast_four_needs_k_major_a(gemm_lib):
    import ctypes
    cfg = gemm_lib._config({"block_n": 64, "multicast": 4})
    h = ctypes.c_void_p()
    lib = gemm_lib.library()
    for layout in (2, 3):                 # TT, NT: A stored K x M
        assert lib.gemm_plan_create_with_config(512, 512, 512, 0, layout, ctypes.byref(cfg),
                                                ctypes.byref(h)) == 1   # INVALID_ARG


def _raster_reference(mb, nb, g, t):
    """The raster order by definition: bands of g m-blocks (the last band may be
    shorter); inside a band the m index runs fastest."""
    band = g * nb
    first_m = (t // band) * g
    r = t % band
    gsize = min(g, mb - first_m)
    return first_m + r % gsize, r // gsize


@pytest.mark.parametrize("mb,nb,g", [(1, 1, 1), (3, 5, 2), (7, 3, 16), (64, 32, 16), (33, 57, 8),
                                     (1000, 3, 7), (4096, 2048, 24), (129, 1, 128), (5, 9, 5),
                                     (46341, 46340, 3)])
def test_raster_matches_its_definition(gemm_lib, mb, nb, g):
    """The kernels evaluate the raster with multiply-shift divisions; compare
    with integer division on tiles spread over the whole grid (both band kinds,
    the last band, large tile ids)."""
    import random
    total = mb * nb
    rng = random.Random(mb * 1000003 + nb * 7 + g)
    ts = set(range(min(total, 2000)))
    ts |= {total - 1 - i for i in range(min(total, 2000))}
    ts |= {rng.randrange(total) for _ in range(3000)}
    for t in sorted(ts):
        assert gemm_lib.gemm_tile_coords(mb, nb, g, t) == _raster_reference(mb, nb, g, t), (t,)


def test_tuner_proposes_only_configs_the_library_accepts(gemm_lib):
    """Every candidate the sweep tuner times, for every sweep and named shape, passes
    the library's own validation (the tuner does not catch plan errors)."""
    from dense_gemm_hgemm_gb300 import tune
    shapes = [(w.M, w.N, w.K, w.dtype) for w in workloads.NAMED + tuple(workloads.sweep_shapes())]
    n = 0
    for M, N, K, dt in shapes:
        for c in tune.candidates(M, N, K, dt, 152):
            gemm_lib.gemm_workspace_bytes(M, N, K, dt, c)   # raises on a rejected config
            n += 1
    assert n > 10000


def test_plan_runner_falls_back_to_the_general_path(gemm_lib):
    """The C-level runner a Plan binds for run(A, B, C, stream) hands every call it
    does not take itself (a closed plan, other argument counts, keywords) to the
    general path with the same arguments; no GPU call is made here."""
    gemm_lib.library()
    pc = gemm_lib._pycall
    if pc is None or not hasattr(pc, "Runner"):
        pytest.skip("CPython entry points not built")
    seen = []

    def general(*args, **kwargs):
        seen.append((args, kwargs))
        return "general"

    class T:
        def data_ptr(self):
            return 256

    class S:
        cuda_stream = 0

    r = pc.Runner([None], general)                     # a closed plan
    t, s = T(), S()
    assert r(t, t, t, s) == "general" and seen[-1] == ((t, t, t, s), {})
    assert r(t, t, t) == "general" and seen[-1] == ((t, t, t), {})
    assert r(t, t, t, s, bias=None) == "general" and seen[-1] == ((t, t, t, s), {"bias": None})
    with pytest.raises(TypeError):
        pc.Runner([], general)
    with pytest.raises(TypeError):
        pc.Runner([None], 5)
