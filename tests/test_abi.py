"""The C-ABI library: it loads, exports every declared symbol, and its host-side
encoders match the PTX ISA field layouts and the pages' worked example.
No GPU is used: only host functions and argument checks are called."""
import os
import re

import pytest

from dense_fp16_gemm_02_gb300 import build, wgemm

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


@pytest.fixture(scope="session")
def lib():
    build.build()
    return wgemm.load()


def _golden(name):
    vals = {}
    for line in open(os.path.join(GOLDEN, name)):
        line = line.strip()
        if line and not line.startswith("#"):
            k, v = line.split()
            vals[k] = int(v, 0)
    return vals


def test_exports_every_declared_function(lib):
    names = wgemm.header_functions()
    assert "wgemm_f16f32" in names and len(names) >= 14
    for n in names:
        assert hasattr(lib, n), n


def test_config_table(lib):
    names = wgemm.config_names()
    assert len(names) == lib.wgemm_num_configs() >= 8
    assert len(set(names)) == len(names)
    assert lib.wgemm_config_name(-1) == b"" and lib.wgemm_config_name(len(names)) == b""
    assert any(n.startswith("g1_") for n in names) and any(n.startswith("g2_") for n in names)


def test_smem_descriptor_worked_example(lib):
    g = _golden("umma_desc_sw128_128x64.txt")
    for addr in (0, 1024, 49152, 200704):
        desc = lib.wgemm_debug_smem_desc(addr)
        assert desc >> 32 == g["high_word"]
        assert (desc & 0x3FFF) == addr >> 4          # start address field
        assert ((desc >> 32) & 0x3FFF) == g["sbo_bytes"] >> 4


def test_smem_descriptor_k_advance(lib):
    # Stepping K by 16 fp16 elements (32 bytes) inside the swizzle row moves
    # only the start-address field, by 2 (16-byte units).
    base = 3 * 1024
    for j in range(4):
        d0, d1 = lib.wgemm_debug_smem_desc(base), lib.wgemm_debug_smem_desc(base + 32 * j)
        assert d1 - d0 == 2 * j


def test_smem_descriptor_offsets_do_not_carry(lib):
    # The MMA thread encodes one descriptor per stage and adds each operand
    # slice's offset in 16-byte units. That equals encoding the slice's own
    # address whenever the sum stays below 256 KB (shared memory per CTA is
    # at most 227 KB): the 14-bit address field never carries.
    for base in range(0, 232 * 1024, 8 * 1024):
        d0 = lib.wgemm_debug_smem_desc(base)
        for off in (16, 32, 96, 1024, 16384, 24 * 1024 + 32, 65536 + 96, 200 * 1024):
            if base + off < 256 * 1024:
                assert lib.wgemm_debug_smem_desc(base + off) == d0 + (off >> 4), (base, off)
    # At 256 KB the field would wrap: the bound is real.
    assert lib.wgemm_debug_smem_desc(256 * 1024) != lib.wgemm_debug_smem_desc(0) + (1 << 14)


def test_sw128_layout_matches_address_bit_xor(lib):
    # TMA's 128-byte swizzle: within each 1024-byte block, byte address bits
    # [4:6] are XORed with bits [7:9]. Rebuild the image of a 128×64 fp16 tile
    # from that rule and compare with the kernels' offset function everywhere.
    seen = set()
    for row in range(128):
        for k in range(64):
            linear = row * 128 + k * 2
            swz = linear ^ (((linear >> 7) & 7) << 4)
            off = lib.wgemm_debug_sw128_offset(row, k)
            assert off == swz
            seen.add(off)
    assert len(seen) == 128 * 64  # a bijection onto the tile's bytes (2-byte steps)


@pytest.mark.parametrize("bf16", [0, 1])
@pytest.mark.parametrize("M,N", [(128, 256), (128, 64), (256, 256), (256, 128), (128, 16)])
def test_instruction_descriptor_fields(lib, M, N, bf16):
    d = lib.wgemm_debug_idesc(M, N, bf16)
    assert (d >> 4) & 3 == 1            # D = f32
    assert (d >> 7) & 7 == bf16 and (d >> 10) & 7 == bf16  # A, B: 0 = f16, 1 = bf16
    assert (d >> 13) & 0xF == 0         # no negation, both K-major
    assert (d >> 17) & 0x3F == N >> 3
    assert (d >> 24) & 0x1F == M >> 4
    assert d & 0xF == 0 and (d >> 23) & 1 == 0 and (d >> 29) == 0


def _call(lib, A, B, C, M, N, K, lda, ldb, ldc):
    return lib.wgemm_f16f32(A, B, C, M, N, K, lda, ldb, ldc, None)


def test_argument_checks_without_launch(lib):
    ok = 1 << 20  # a 16-byte aligned stand-in address; rejected calls never touch it
    assert _call(lib, ok, ok, ok, -1, 4, 4, 8, 8, 4) == -1
    assert _call(lib, ok, ok, ok, 4, 4, -1, 8, 8, 4) == -1
    assert _call(lib, None, ok, ok, 4, 4, 8, 8, 8, 4) == -1
    assert _call(lib, ok, ok, None, 4, 4, 8, 8, 8, 4) == -1
    assert _call(lib, ok, ok, ok, 4, 4, 16, 8, 16, 4) == -1     # lda < K
    assert _call(lib, ok, ok, ok, 4, 4, 8, 8, 8, 2) == -1       # ldc < N
    assert _call(lib, ok + 2, ok, ok, 4, 4, 8, 8, 8, 4) == -2   # A misaligned
    assert _call(lib, ok, ok, ok + 2, 4, 4, 8, 8, 8, 4) == -2   # C not 4-byte aligned
    assert _call(lib, ok, ok, ok, 4, 4, 8, 12, 8, 4) == -2      # lda % 8
    assert _call(lib, None, None, None, 0, 4, 8, 8, 8, 4) == 0  # empty: no-op
    assert _call(lib, None, None, None, 4, 0, 8, 8, 8, 4) == 0


def test_status_strings(lib):
    for code in range(-7, 1):
        s = lib.wgemm_status_string(code).decode()
        assert s and s != "unknown status"
    assert lib.wgemm_status_string(-99).decode() == "unknown status"


def test_rule_predictions_from_measured_rates(lib):
    """The per-shape rule's host arithmetic: every configuration has measured
    rates, predictions grow with K and with waves of tiles, and invalid
    arguments give -1."""
    n = lib.wgemm_num_configs()
    for cid in range(n):
        name = lib.wgemm_config_name(cid).decode()
        w = 36 if re.match(r"g2[mr]2_", name) else (152 if name.startswith("g1_") else 76)
        p = lambda M, N, K, ld=None, mode=0, s=1: lib.wgemm_debug_predict_us(
            M, N, K, ld or K, ld or K, cid, mode, s, w)
        assert p(4096, 4096, 2048) > 0, name
        assert p(4096, 4096, 4096) > p(4096, 4096, 2048), name
        assert p(16384, 16384, 2048) > p(4096, 4096, 2048), name
        assert p(4096, 4096, 2048, ld=2056) > 0, name
        assert p(4096, 4096, 2048, ld=1024) == -1.0, name  # pitch below K
    assert lib.wgemm_debug_predict_us(64, 64, 64, 64, 64, n, 0, 1, 76) == -1.0
    assert lib.wgemm_debug_predict_us(64, 64, 64, 64, 64, -1, 0, 1, 76) == -1.0
    # The waves + stream-K tail mix is not modelled.
    cid = wgemm.config_id("g2_256x256_s6_a2_tma")
    assert lib.wgemm_debug_predict_us(4096, 4096, 4096, 4096, 4096, cid, 3, 1, 76) == -1.0


def test_rule_charges_rows_off_sectors(lib):
    """Rows 16 bytes off 32-byte sectors cost 256-column pair tiles more than a
    fifth more time at 3000×5000×3000 (measured), and the prediction says so."""
    cid = wgemm.config_id("g2_256x224_s7_a2_direct")
    on = lib.wgemm_debug_predict_us(3000, 5000, 3000, 3008, 3008, cid, 0, 1, 76)
    off = lib.wgemm_debug_predict_us(3000, 5000, 3000, 3000, 3000, cid, 0, 1, 76)
    assert off > 1.1 * on > 0


def test_typed_entry_points_check_arguments_without_launch(lib):
    ok = 1 << 20
    F32, F16, BF16 = wgemm.WGEMM_F32, wgemm.WGEMM_F16, wgemm.WGEMM_BF16
    g = lambda A, B, C, ab, c, ldc=8: lib.wgemm_gemm(A, B, C, ab, c, 4, 4, 8, 8, 8, ldc, None)
    assert g(ok, ok, ok, F32, F32) == -1          # fp32 operands: not a tensor-core type here
    assert g(ok, ok, ok, 3, F32) == -1
    assert g(ok, ok, ok, F16, 7) == -1
    assert g(ok, ok, ok + 1, F16, F16) == -2      # 16-bit C must be 2-byte aligned
    assert g(ok, ok, ok + 2, BF16, F32) == -2     # fp32 C must be 4-byte aligned
    assert g(ok, ok, ok, BF16, BF16, ldc=2) == -1  # ldc < N
    assert lib.wgemm_gemm(None, None, None, F16, BF16, 0, 4, 8, 8, 8, 4, None) == 0
    for fn in (lib.wgemm_bf16f32, lib.wgemm_f16f16, lib.wgemm_bf16bf16):
        assert fn(ok, ok, ok, -1, 4, 8, 8, 8, 4, None) == -1


def test_configurations_name_their_c_width(lib):
    names = wgemm.config_names()
    outs = [lib.wgemm_debug_config_out(i) for i in range(len(names))]
    assert all(o == (1 if n.endswith("_h") else 0) for n, o in zip(names, outs))
    assert 0 in outs and 1 in outs
    assert lib.wgemm_debug_config_out(len(names)) == -6
    # every plain 16-bit configuration is an fp32 configuration with another
    # epilogue; fused configurations say so in their name
    fused = [lib.wgemm_debug_config_fused(i) for i in range(len(names))]
    assert all(f == (1 if "_ab" in n else 0) for n, f in zip(names, fused))
    assert 1 in fused and lib.wgemm_debug_config_fused(len(names)) == -6
    for n in names:
        if n.endswith("_h") and "_ab" not in n:
            assert n[:-2] in names


def test_cooperative_switch(lib):
    # Host-only: the profiling hook toggles the cooperative attribute of
    # K-split launches; the default is on.
    assert lib.wgemm_debug_set_cooperative(2) == -1 and lib.wgemm_debug_set_cooperative(-1) == -1
    assert lib.wgemm_debug_set_cooperative(0) == 1
    assert lib.wgemm_debug_set_cooperative(1) == 0
    assert lib.wgemm_debug_set_cooperative(1) == 1


def test_pdl_switch(lib):
    assert lib.wgemm_set_pdl(2) == -1 and lib.wgemm_set_pdl(-1) == -1
    prev = lib.wgemm_set_pdl(1)
    assert prev in (0, 1)
    assert lib.wgemm_set_pdl(0) == 1
    assert lib.wgemm_set_pdl(prev) == 0


def test_peak_microbenchmark_compiles():
    """The tensor-pipe microbenchmark (peak/tensor_peak.cu) builds for sm_103a."""
    from dense_fp16_gemm_02_gb300 import peak
    exe = peak.build_peak("tensor_peak")
    assert os.path.exists(exe) and os.access(exe, os.X_OK)


def test_ncu_summary_maps_every_configuration_to_its_template_arguments(tmp_path):
    import ncu_summary
    names = wgemm.config_names()
    args = [ncu_summary._entry_args(n) for n in names]
    assert all(a is not None and len(a) == 12 for a in args)
    assert len(set(args)) == len(names)  # one configuration per template instantiation
    kernel = "void wgemm_kernel<Cfg<%s>>(KParams)" % ", ".join(str(x) for x in args[0])
    assert ncu_summary._config_of_kernel(kernel) == names[0]
    # A row-multicast configuration, one with two k-blocks per stage, and
    # names captured before the eleventh and twelfth template arguments existed.
    for pick in ([n for n in names if "r2_" in n][0], [n for n in names if "x2_a" in n][0]):
        k = "void wgemm_kernel<Cfg<%s>>(KParams)" % ", ".join(str(x) for x in args[names.index(pick)])
        assert ncu_summary._config_of_kernel(k) == pick
    assert ncu_summary._entry_args("g1_128x64_s4x2_a2_direct")[-1] == 2
    for n_args in (10, 11):
        old = "void wgemm_kernel<Cfg<%s>>(KParams)" % ", ".join(str(x) for x in args[0][:n_args])
        assert ncu_summary._config_of_kernel(old) == names[0]
    csv_text = ('"ID","Process ID","Process Name","Host Name","Kernel Name","Context","Stream",'
                '"Block Size","Grid Size","Device","CC","Section Name","Metric Name","Metric Unit",'
                '"Metric Value"\n'
                '"0","1","python","h","%s","1","7","(256, 1, 1)","(152, 1, 1)","0","10.3","",'
                '"gpu__time_duration.sum","ns","13,312"\n' % kernel)
    p = tmp_path / "x.csv"
    p.write_text("==PROF== preamble\n" + csv_text)
    by = ncu_summary.read_ncu_csv(str(p))
    assert by["0"]["gpu__time_duration.sum"] == 13312.0 and by["0"]["kernel"] == kernel


def test_ncu_summary_warm_groups_launches_by_arm_and_call(tmp_path, capsys):
    # compare --warm runs, per shape, the library's calls and then cuBLAS's;
    # a cuBLAS call may launch several kernels, summed per call; the first
    # three calls of each arm are warm-up. A start-up probe before the first
    # library launch is skipped.
    import ncu_summary
    head = ('"ID","Process ID","Process Name","Host Name","Kernel Name","Context","Stream",'
            '"Block Size","Grid Size","Device","CC","Metric Name","Metric Unit","Metric Value"')
    rows, n = [], 0

    def add(kernel, us):
        nonlocal n
        rows.append(f'"{n}","1","python","h","{kernel}","1","7","(256, 1, 1)","(1, 1, 1)",'
                    f'"0","10.3","gpu__time_duration.sum","ns","{int(us * 1000)}"')
        n += 1

    add("nvjet_probe", 50.0)
    for s in range(2):
        for c in range(5):  # 3 warm-up + 2 timed library calls
            add("void wg::wgemm_kernel<wg::Cfg<1>>(wg::KParams)", 100.0 if c < 3 else 10.0 + s)
        for c in range(5):  # cuBLAS: two kernels per call
            add("nvjet_main", 100.0 if c < 3 else 5.0 + s)
            add("nvjet_reduce", 1.0)
    (tmp_path / "w.csv").write_text(head + "\n" + "\n".join(rows) + "\n")
    (tmp_path / "c.jsonl").write_text(
        '{"shape": "64x64x64", "ours_us": 12.0, "cublas_us": 9.0}\n'
        '{"shape": "128x64x64", "ours_us": 13.0, "cublas_us": 10.0}\n'
        '{"summary": {"rounds": 2}}\n')
    ncu_summary.warm(str(tmp_path / "w.csv"), str(tmp_path / "c.jsonl"))
    out = [l for l in capsys.readouterr().out.splitlines() if l.startswith("| 6") or
           l.startswith("| 1")]
    assert out[0].startswith("| 64×64×64 | 10.00 | 6.00 | 0.600 |")
    assert out[1].startswith("| 128×64×64 | 11.00 | 7.00 | 0.636 |")
    assert "| 2 |" in out[0]


def test_host_buffer_entry_without_launch(lib):
    """wgemm_f16f32_host checks its arguments before it touches a device, and
    the device buffer sizes and the panel rule are host arithmetic."""
    call = wgemm.wgemm_f16f32_host
    h, d = 4096, 4096  # stand-in addresses, never dereferenced here
    assert call(h, h, h, -1, 4, 8, 8, 8, 4, d, d, d, None) == -1
    assert call(h, h, h, 0, 4, 8, 8, 8, 4, d, d, d, None) == 0  # nothing to do
    assert call(h, h, None, 4, 4, 8, 8, 8, 4, d, d, d, None) == -1  # no host C
    assert call(h, h, h, 4, 4, 8, 8, 8, 3, d, d, d, None) == -1  # ldc < N
    assert call(None, h, h, 4, 4, 8, 8, 8, 4, d, d, d, None) == -1  # no host A
    assert call(h, h, h, 4, 4, 8, 8, 8, 4, d + 8, d, d, None) == -2  # device A off 16 B
    assert call(h, h, h, 4, 4, 8, 8, 8, 4, d, d, d + 4, None) == -2  # device C off 16 B
    # Device pitches: K up to a multiple of 8, N up to a multiple of 4.
    assert wgemm.host_device_elems(600, 1101, 300) == (600 * 304, 1101 * 304, 600 * 1104)
    assert wgemm.host_device_elems(0, 0, 0) == (0, 0, 0)
    with pytest.raises(ValueError):
        wgemm.host_device_elems(-1, 4, 4)
    # Panels: min(A bytes, C bytes) / 8 MiB, 1 to 8, rows a multiple of 256.
    rows = lib.wgemm_debug_host_panel_rows
    assert rows(16384, 16384, 16384) == 2048
    assert rows(8192, 8192, 8192) == 1024
    assert rows(4096, 4096, 4096) == 1024  # A is 32 MiB: four panels
    assert rows(2048, 2048, 2048) == 2048  # A is 8 MiB: one panel
    assert rows(1024, 1024, 65536) == 1024  # C is 4 MiB: one panel
    assert rows(600, 1100, 300) == 600
    assert rows(0, 4, 4) == -1
    prev = lib.wgemm_debug_set_host_panels(3)
    try:
        assert rows(1000, 777, 520) == 512  # ceil(1000 / 3) rounded up to 256
    finally:
        lib.wgemm_debug_set_host_panels(prev)
    assert lib.wgemm_debug_set_host_panels(9) == -1
    # Blocks of B's rows (C's columns): B bytes / 128 MiB, 1 to 4, a multiple
    # of 256 rows each.
    cols = lib.wgemm_debug_host_block_cols
    assert cols(16384, 16384) == 4096  # B is 512 MiB: four blocks
    assert cols(8192, 8192) == 8192  # 128 MiB: one block
    assert cols(8192, 32768) == 2048  # 512 MiB: four blocks
    assert cols(2048, 65536) == 1024  # 256 MiB: two blocks
    assert cols(1024, 65536) == 1024  # 128 MiB: one block
    assert cols(777, 520) == 777
    assert cols(0, 4) == -1 and cols(4, 0) == -1
    prev = lib.wgemm_debug_set_host_blocks(2)
    try:
        assert cols(777, 520) == 512  # ceil(777 / 2) rounded up to 256
        assert cols(200, 520) == 200  # one block of 256 covers it
        lib.wgemm_debug_set_host_blocks(4)
        assert cols(777, 520) == 256  # 256 + 256 + 256 + 9
    finally:
        lib.wgemm_debug_set_host_blocks(prev)
    assert lib.wgemm_debug_set_host_blocks(5) == -1
    assert lib.wgemm_debug_set_host_blocks(-1) == -1
