"""Write the operator pages' worked examples as JSON fixtures beside this script.

Usage:  python tests/golden/extract_page_examples.py <pages.txt> [out_dir]

<pages.txt> is the plain-text capture of the operator pages (AffineGrid,
Resize, GridSample - version 20, DeformConv, GridSample).  The script only
transcribes the numbers the pages print -- inputs, attributes and expected
outputs -- into one fixture per example; it computes nothing.  Each fixture
carries a ``citation`` naming the page and the example it came from, and a
``notes`` field for anything the page left out (elided channels, defaults).

The fixtures are committed; the tests read only the fixtures, never the pages.
"""
import json
import os
import re
import sys

import numpy as np

# (page title used in citations, example marker regex, example name)
AFFINE = "AffineGrid (ai.onnx, since version 20)"
GRIDSAMPLE = "GridSample - version 20"
DEFORM = "DeformConv (ai.onnx, since version 22)"
RESIZE = "Resize - 18 (mlprodict operator page)"

AFFINE_NAMES = ["test_affine_grid_2d", "test_affine_grid_2d_align_corners",
                "test_affine_grid_3d", "test_affine_grid_3d_align_corners"]
GRIDSAMPLE_NAMES = [
    "test_gridsample", "test_gridsample_aligncorners_true",
    "test_gridsample_bicubic", "test_gridsample_bicubic_align_corners_0_additional_1",
    "test_gridsample_bicubic_align_corners_1_additional_1", "test_gridsample_bilinear",
    "test_gridsample_bilinear_align_corners_0_additional_1",
    "test_gridsample_bilinear_align_corners_1_additional_1", "test_gridsample_border_padding",
    "test_gridsample_nearest", "test_gridsample_nearest_align_corners_0_additional_1",
    "test_gridsample_nearest_align_corners_1_additional_1", "test_gridsample_reflection_padding",
    "test_gridsample_volumetric_bilinear_align_corners_0",
    "test_gridsample_volumetric_bilinear_align_corners_1",
    "test_gridsample_volumetric_nearest_align_corners_0",
    "test_gridsample_volumetric_nearest_align_corners_1", "test_gridsample_zeros_padding",
]
DEFORM_NAMES = ["test_cc_basic_deform_conv_with_padding",
                "test_cc_basic_deform_conv_without_padding",
                "test_cc_deform_conv_with_mask_bias",
                "test_cc_deform_conv_with_multiple_offset_groups"]
# Resize: every example on the page (found by name in main()); the ones
# listed here were the first transcribed and keep their fixture names.
RESIZE_MARKER = re.compile(r"\*\*(_resize_[A-Za-z0-9_]+)\*\*")

NUM = re.compile(r"-?\d+\.\d*(?:[eE][-+]?\d+)?|-?\d+(?:[eE][-+]?\d+)?|-?\.\d+")


def balanced(text, start):
    """Return the bracket-balanced substring of ``text`` starting at the first '[' at or after start."""
    i = text.index("[", start)
    depth = 0
    for j in range(i, len(text)):
        ch = text[j]
        if ch == "[":
            depth += 1
        elif ch == "]":
            depth -= 1
            if depth == 0:
                return text[i:j + 1], j + 1
    raise ValueError("unbalanced brackets")


def nested(text):
    """Parse '[[1, 2], [3 4]]' (commas optional, '#' ignored) into nested lists."""
    toks = re.findall(r"\[|\]|" + NUM.pattern, text.replace("#", " "))
    stack = [[]]
    for t in toks:
        if t == "[":
            stack.append([])
        elif t == "]":
            top = stack.pop()
            stack[-1].append(top)
        else:
            stack[-1].append(float(t))
    return stack[0][0]


def tensor_entry(shape, dtype, flat, note=None):
    e = {"shape": list(shape), "dtype": dtype, "data": [float(v) for v in flat]}
    if note:
        e["note"] = note
    return e


def parse_onnx_tensors(seg):
    """Tensors printed as 'name: shape=(...), dtype=...' followed by a bracketed array."""
    out = {}
    notes = []
    for m in re.finditer(r"(\w+): shape=\(([^)]*)\), dtype=(\w+)", seg):
        name, shp, dt = m.group(1), m.group(2), m.group(3)
        shape = [int(s) for s in shp.replace(" ", "").split(",") if s]
        body, _ = balanced(seg, m.end())
        count = int(np.prod(shape)) if shape else 1
        if "..." in body:
            # The page elides whole channel blocks of a batch-1 tensor with '...'.
            before, after = body.split("...")
            a = [float(v) for v in NUM.findall(before)]
            b = [float(v) for v in NUM.findall(after)]
            block = int(np.prod(shape[2:]))
            assert shape[0] == 1 and len(a) % block == 0 and len(b) % block == 0
            missing = count - len(a) - len(b)
            first = len(a) // block
            nmiss = missing // block
            note = (f"channels {first}..{first + nmiss - 1} are elided on the page ('...'); "
                    "read as zeros")
            notes.append(f"{name}: {note}")
            flat = a + [0.0] * missing + b
            out[name] = tensor_entry(shape, dt, flat, note)
        else:
            flat = [float(v) for v in NUM.findall(body)]
            assert len(flat) == count, (name, len(flat), count)
            out[name] = tensor_entry(shape, dt, flat)
    return out, notes


def parse_onnx_attributes(seg):
    m = re.search(r"Attributes:(.*?)(?:Inputs:|\.\. code-block)", seg, re.S)
    attrs = {}
    if not m:
        return attrs
    for k, v in re.findall(r"(\w+)\s*=\s*(\"[^\"]*\"|\[[^\]]*\]|-?[\d.]+)", m.group(1)):
        if v.startswith('"'):
            attrs[k] = v.strip('"')
        elif v.startswith("["):
            attrs[k] = [int(x) for x in NUM.findall(v)]
        else:
            attrs[k] = float(v) if "." in v else int(v)
    return attrs


def segments(text, names, marker):
    """Slice ``text`` into one segment per example name, in page order."""
    pos = []
    for n in names:
        m = re.search(marker(n), text, re.M)
        assert m, n
        pos.append((m.start(), n))
    pos.sort()
    segs = {}
    for i, (p, n) in enumerate(pos):
        end = pos[i + 1][0] if i + 1 < len(pos) else len(text)
        nxt = text.find("=-=-= page", p)
        if nxt != -1:
            end = min(end, nxt)
        segs[n] = text[p:end]
    return segs


def onnx_fixture(op, page, name, seg):
    tensors, notes = parse_onnx_tensors(seg)
    split = seg.index("Outputs:")
    outs = {}
    ins = {}
    for k, v in tensors.items():
        hdr = seg.index(f"{k}: shape=")
        (outs if hdr > split else ins)[k] = v
    node = re.search(r"Node:\s*(\w+\([^)]*\)\s*->\s*\([^)]*\))", seg)
    return {"citation": f"{page}, Examples, {name}", "op": op, "name": name,
            "node": node.group(1) if node else None,
            "attributes": parse_onnx_attributes(seg), "inputs": ins, "outputs": outs,
            "notes": notes}


def _resize_value(v, env):
    """A make_node keyword value: a literal, or a variable assigned earlier in the example."""
    if v.startswith('"'):
        return v.strip('"')
    if v in ("True", "False"):
        return int(v == "True")
    if re.fullmatch(r"-?[\d.]+", v):
        return float(v) if "." in v else int(v)
    return env[v]


def resize_fixture(name, seg):
    # variables the example assigns before make_node (axes, keep_aspect_ratio_policy)
    env = {}
    head = seg[:seg.index("make_node(")]
    for k, v in re.findall(r"(\w+)\s*=\s*(\"[^\"]*\"|\[[^\]]*\])", head):
        env[k] = v.strip('"') if v.startswith('"') else [int(x) for x in NUM.findall(v)]
    attrs = {}
    node = re.search(r"make_node\((.*?)\)\s*data", seg, re.S).group(1)
    for k, v in re.findall(r"(\w+)=(\"[^\"]*\"|-?[\d.]+|True|False|[A-Za-z_]\w*)", node):
        if k in ("inputs", "outputs"):
            continue
        attrs[k] = _resize_value(v, env)
    data_txt, _ = balanced(seg, seg.index("data = np.array("))
    data = np.array(nested(data_txt), dtype=np.float64)
    ins = {"X": tensor_entry(data.shape, "float32", data.ravel())}
    m = re.search(r"\broi = np\.array\(", seg)
    if m:
        roi_txt, _ = balanced(seg, m.end() - 1)
        roi = [float(v) for v in NUM.findall(roi_txt)]
        ins["roi"] = tensor_entry([len(roi)], "float32", roi)
    m = re.search(r"(scales|sizes) = np\.array\(", seg)
    vec_txt, vec_end = balanced(seg, m.end() - 1)
    vec = [float(v) for v in NUM.findall(vec_txt)]
    if m.group(1) == "scales":
        ins["scales"] = tensor_entry([len(vec)], "float32", vec)
    else:
        ins["sizes"] = tensor_entry([len(vec)], "int64", vec)
    exp_txt, _ = balanced(seg, seg.index("# [", vec_end) + 2)
    exp = np.array(nested(exp_txt), dtype=np.float64)
    fx = {"citation": f"{RESIZE}, Examples, {name}", "op": "Resize", "name": name,
          "attributes": attrs, "inputs": ins,
          "outputs": {"Y": tensor_entry(exp.shape, "float32", exp.ravel())},
          "notes": ["expected output is the array printed in the example's comment"]}
    # some examples state the output extent in words ("# Results in 8x8")
    m = re.search(r"# Results in (\d+)x(\d+)", seg[vec_end:])
    if m:
        stated = [int(m.group(1)), int(m.group(2))]
        fx["stated_spatial_shape"] = stated
        if list(exp.shape[-2:]) != stated:
            fx["notes"].append(f"the page states {stated[0]}x{stated[1]} but prints "
                               f"{exp.shape[-2]}x{exp.shape[-1]}: the printed rows are read as "
                               "the first rows of the stated output")
    return fx


def main():
    src = sys.argv[1]
    out_dir = sys.argv[2] if len(sys.argv) > 2 else os.path.dirname(os.path.abspath(__file__))
    with open(src, encoding="utf-8") as f:
        text = f.read()
    fixtures = []
    for n, seg in segments(text, AFFINE_NAMES, lambda n: rf"^{re.escape(n)}\s*$").items():
        fixtures.append(onnx_fixture("AffineGrid", AFFINE, n, seg))
    for n, seg in segments(text, GRIDSAMPLE_NAMES, lambda n: rf"\*\*{re.escape(n)}\*\*").items():
        fixtures.append(onnx_fixture("GridSample", GRIDSAMPLE, n, seg))
    for n, seg in segments(text, DEFORM_NAMES, lambda n: rf"\*\*{re.escape(n)}\*\*").items():
        fixtures.append(onnx_fixture("DeformConv", DEFORM, n, seg))
    resize_names = list(dict.fromkeys(RESIZE_MARKER.findall(text)))
    for n, seg in segments(text, resize_names, lambda n: rf"\*\*{re.escape(n)}\*\*").items():
        fixtures.append(resize_fixture(n, seg))
    for fx in fixtures:
        path = os.path.join(out_dir, f"{fx['op'].lower()}__{fx['name'].lstrip('_')}.json")
        with open(path, "w") as f:
            json.dump(fx, f, indent=1)
            f.write("\n")
    print(f"wrote {len(fixtures)} fixtures to {out_dir}")


if __name__ == "__main__":
    main()
