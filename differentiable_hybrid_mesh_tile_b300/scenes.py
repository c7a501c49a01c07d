"""Seeded synthetic scenes for the hybrid mesh + 3D Gaussian renderer.

This module only draws inputs: camera poses, triangle meshes with vertex
colours, and 3D Gaussians in the stored parameterisation (means, log-scales,
quaternions, opacity logits, colours).  It holds none of the renderer's
arithmetic, so both the CUDA path and the CPU oracle can take their inputs
from it.

The five workloads follow the hybrid-rendering setting of "A Lightweight and
Differentiable Renderer for Joint Mesh and 3D Gaussian Splat Scenes"
(Design Details: one pinhole camera shared by mesh and Gaussians, a mesh with
vertex colours, Gaussians with means / rotations / scales / opacities /
colours).  The stored Gaussian parameterisation (opacity as a logit, scale as
a log, rotation as a quaternion, SH DC colour) is the one listed in the
"Gaussian splatting reference" page, section "Output writing".

Conventions (readings, stated once here):
  * camera frame is the OpenCV one: x right, y down, z forward;
    ``R`` (row-major 3x3) and ``t`` map world to camera: X_c = R X_w + t;
  * look-at uses world up (0, 1, 0), or (0, 0, 1) when the view direction is
    within 0.999 of it;
  * pixel (i, j) has its centre at (i + 0.5, j + 0.5);
  * quaternions are (w, x, y, z);
  * ``sh_degree == -1`` means the colours are plain RGB [N, 3]; degree d >= 0
    means [N, (d + 1)^2, 3] real SH coefficients.

Every array is drawn from ``numpy.random.default_rng(seed)`` in the order the
generator functions list, so a seed fixes the scene bit for bit.
"""

from __future__ import annotations

import dataclasses
import math
from typing import List, Optional

import numpy as np

TILE = 16
NEAR = 0.01
FAR = 1.0e10
BG_WHITE = (1.0, 1.0, 1.0)


@dataclasses.dataclass
class Camera:
    width: int
    height: int
    fx: float
    fy: float
    cx: float
    cy: float
    near: float
    far: float
    R: np.ndarray  # [3, 3] float32, world -> camera
    t: np.ndarray  # [3] float32

    @property
    def tiles_x(self) -> int:
        return (self.width + TILE - 1) // TILE

    @property
    def tiles_y(self) -> int:
        return (self.height + TILE - 1) // TILE

    @property
    def n_tiles(self) -> int:
        return self.tiles_x * self.tiles_y


@dataclasses.dataclass
class Mesh:
    verts: np.ndarray   # [V, 3] float32 world positions
    faces: np.ndarray   # [F, 3] int32 vertex indices
    vcol: np.ndarray    # [V, 3] float32 RGB


@dataclasses.dataclass
class Gaussians:
    means: np.ndarray       # [N, 3] float32
    log_scales: np.ndarray  # [N, 3] float32
    quats: np.ndarray       # [N, 4] float32, (w, x, y, z)
    logits: np.ndarray      # [N] float32 opacity logits
    colors: np.ndarray      # [N, 3] RGB or [N, (d+1)^2, 3] SH coefficients
    sh_degree: int          # -1 = RGB


@dataclasses.dataclass
class Scene:
    name: str
    cameras: List[Camera]
    mesh: Mesh
    gaussians: Gaussians
    bg: tuple = BG_WHITE

    @property
    def camera(self) -> Camera:
        return self.cameras[0]


# ----------------------------------------------------------------------------
# cameras
# ----------------------------------------------------------------------------

def look_at(eye, target, width, height, fx, fy, cx=None, cy=None,
            near=NEAR, far=FAR) -> Camera:
    eye = np.asarray(eye, np.float64)
    target = np.asarray(target, np.float64)
    fwd = target - eye
    fwd /= np.linalg.norm(fwd)
    up = np.array([0.0, 1.0, 0.0])
    if abs(float(fwd @ up)) > 0.999:
        up = np.array([0.0, 0.0, 1.0])
    right = np.cross(fwd, up)
    right /= np.linalg.norm(right)
    down = np.cross(fwd, right)
    R = np.stack([right, down, fwd], 0)
    t = -R @ eye
    return Camera(width=int(width), height=int(height), fx=float(fx), fy=float(fy),
                  cx=float(width / 2 if cx is None else cx),
                  cy=float(height / 2 if cy is None else cy),
                  near=float(near), far=float(far),
                  R=R.astype(np.float32), t=t.astype(np.float32))


# ----------------------------------------------------------------------------
# meshes
# ----------------------------------------------------------------------------

def icosahedron():
    """12 vertices on the unit sphere and the 20 faces, outward-oriented.

    Faces are found as the triples of mutually adjacent vertices (adjacent =
    at the edge length of the (+-1, +-phi, 0) construction)."""
    phi = (1.0 + math.sqrt(5.0)) / 2.0
    v = []
    for a in (-1.0, 1.0):
        for b in (-phi, phi):
            v += [(a, b, 0.0), (0.0, a, b), (b, 0.0, a)]
    v = np.array(v, np.float64)
    d = np.linalg.norm(v[:, None, :] - v[None, :, :], axis=-1)
    adj = np.abs(d - 2.0) < 1e-9
    faces = []
    n = len(v)
    for i in range(n):
        for j in range(i + 1, n):
            if not adj[i, j]:
                continue
            for k in range(j + 1, n):
                if adj[i, k] and adj[j, k]:
                    c = v[i] + v[j] + v[k]
                    nrm = np.cross(v[j] - v[i], v[k] - v[i])
                    faces.append((i, j, k) if nrm @ c > 0 else (i, k, j))
    assert len(faces) == 20
    v /= np.linalg.norm(v, axis=1, keepdims=True)
    return v, np.array(faces, np.int64)


def subdivide(v, f):
    """Split every face into four at the edge midpoints, pushed to the unit sphere."""
    e = np.concatenate([f[:, [0, 1]], f[:, [1, 2]], f[:, [2, 0]]], 0)
    e_sorted = np.sort(e, axis=1)
    uniq, inv = np.unique(e_sorted, axis=0, return_inverse=True)
    inv = inv.reshape(-1)
    mid = 0.5 * (v[uniq[:, 0]] + v[uniq[:, 1]])
    mid /= np.linalg.norm(mid, axis=1, keepdims=True)
    nf = len(f)
    m01 = len(v) + inv[:nf]
    m12 = len(v) + inv[nf:2 * nf]
    m20 = len(v) + inv[2 * nf:]
    a, b, c = f[:, 0], f[:, 1], f[:, 2]
    nfaces = np.concatenate([
        np.stack([a, m01, m20], 1),
        np.stack([b, m12, m01], 1),
        np.stack([c, m20, m12], 1),
        np.stack([m01, m12, m20], 1)], 0)
    return np.concatenate([v, mid], 0), nfaces


def icosphere(levels: int):
    v, f = icosahedron()
    for _ in range(levels):
        v, f = subdivide(v, f)
    return v, f


def vertex_neighbour_mean(values, faces, n_verts):
    """Mean of ``values`` over each vertex's 1-ring (edge) neighbours."""
    e = np.concatenate([faces[:, [0, 1]], faces[:, [1, 2]], faces[:, [2, 0]]], 0)
    e = np.unique(np.sort(e, axis=1), axis=0)
    acc = np.zeros(n_verts, np.float64)
    deg = np.zeros(n_verts, np.float64)
    np.add.at(acc, e[:, 0], values[e[:, 1]])
    np.add.at(acc, e[:, 1], values[e[:, 0]])
    np.add.at(deg, e[:, 0], 1.0)
    np.add.at(deg, e[:, 1], 1.0)
    return acc / np.maximum(deg, 1.0)


def triangle_soup(rng, n_tri, centroid_lo, centroid_hi, jitter):
    lo = np.asarray(centroid_lo, np.float64)
    hi = np.asarray(centroid_hi, np.float64)
    cen = rng.uniform(lo, hi, size=(n_tri, 3))
    verts = cen[:, None, :] + rng.normal(0.0, jitter, size=(n_tri, 3, 3))
    verts = verts.reshape(-1, 3)
    faces = np.arange(3 * n_tri, dtype=np.int64).reshape(n_tri, 3)
    return verts, faces


def random_unit(rng, n):
    d = rng.normal(size=(n, 3))
    return d / np.linalg.norm(d, axis=1, keepdims=True)


# ----------------------------------------------------------------------------
# Gaussians
# ----------------------------------------------------------------------------

def _gaussians(rng, means, ls_mu, ls_sd, logit_sd, sh_degree):
    n = len(means)
    log_scales = rng.normal(ls_mu, ls_sd, size=(n, 3))
    q = rng.normal(size=(n, 4))
    q /= np.linalg.norm(q, axis=1, keepdims=True)
    logits = rng.normal(0.0, logit_sd, size=n)
    if sh_degree < 0:
        colors = rng.uniform(0.0, 1.0, size=(n, 3))
    else:
        k = (sh_degree + 1) ** 2
        colors = rng.normal(0.0, 0.2, size=(n, k, 3))
        colors[:, 0, :] = rng.normal(0.5, 0.2, size=(n, 3))
    return Gaussians(means=means.astype(np.float32),
                     log_scales=log_scales.astype(np.float32),
                     quats=q.astype(np.float32),
                     logits=logits.astype(np.float32),
                     colors=np.ascontiguousarray(colors, np.float32),
                     sh_degree=sh_degree)


def _mesh(v, f, vcol):
    return Mesh(verts=np.ascontiguousarray(v, np.float32),
                faces=np.ascontiguousarray(f, np.int32),
                vcol=np.ascontiguousarray(vcol, np.float32))


# ----------------------------------------------------------------------------
# the five workloads
# ----------------------------------------------------------------------------

def tiny(seed: int = 0) -> Scene:
    """64x64 px; once-subdivided icosahedron (42 v / 80 f); 1,000 Gaussians."""
    rng = np.random.default_rng(seed)
    cam = look_at((0, 0, 4), (0, 0, 0), 64, 64, 64, 64, 32, 32)
    v, f = icosphere(1)
    vcol = rng.uniform(0, 1, size=(len(v), 3))
    means = rng.uniform(-1.5, 1.5, size=(1000, 3))
    g = _gaussians(rng, means, -3.0, 0.5, 1.0, -1)
    return Scene("tiny_64", [cam], _mesh(v, f, vcol), g)


def sphere512(seed: int = 1) -> Scene:
    """512x512 px; 4x-subdivided icosphere (2,562 v / 5,120 f); 100k Gaussians."""
    rng = np.random.default_rng(seed)
    eye = 3.5 * random_unit(rng, 1)[0]
    cam = look_at(eye, (0, 0, 0), 512, 512, 512, 512)
    v, f = icosphere(4)
    vcol = rng.uniform(0, 1, size=(len(v), 3))
    n = 100_000
    means = random_unit(rng, n) * rng.uniform(0.8, 1.4, size=(n, 1))
    g = _gaussians(rng, means, -4.0, 0.5, 1.5, -1)
    return Scene("sphere_512", [cam], _mesh(v, f, vcol), g)


def soup1080(seed: int = 2, n_gauss: int = 1_000_000, n_tri: int = 200_000) -> Scene:
    """1920x1080; 200k-triangle soup; 1M Gaussians with SH degree 3."""
    rng = np.random.default_rng(seed)
    cam = look_at((0, 0, 6), (0, 0, 0), 1920, 1080, 1200, 1200)
    v, f = triangle_soup(rng, n_tri, (-2, -2, -2), (2, 2, 2), 0.03)
    vcol = rng.uniform(0, 1, size=(len(v), 3))
    means = rng.uniform(-2.5, 2.5, size=(n_gauss, 3))
    g = _gaussians(rng, means, -4.5, 0.6, 1.5, 3)
    return Scene("soup_1080p", [cam], _mesh(v, f, vcol), g)


def orbit1080(seed: int = 3, n_gauss: int = 3_000_000, levels: int = 7) -> Scene:
    """8 views of 1920x1080 on a radius-5 orbit; displaced 7x icosphere; 3M Gaussians SH3."""
    rng = np.random.default_rng(seed)
    cams = []
    for k in range(8):
        a = 2.0 * math.pi * k / 8.0
        eye = (5.0 * math.cos(a), 0.0, 5.0 * math.sin(a))
        cams.append(look_at(eye, (0, 0, 0), 1920, 1080, 1200, 1200))
    v, f = icosphere(levels)
    nv = rng.normal(size=len(v))
    for _ in range(3):
        nv = vertex_neighbour_mean(nv, f, len(v))
    v = 1.5 * v * (1.0 + (0.1 / 1.5) * nv)[:, None]
    vcol = rng.uniform(0, 1, size=(len(v), 3))
    means = random_unit(rng, n_gauss) * rng.uniform(1.2, 2.2, size=(n_gauss, 1))
    g = _gaussians(rng, means, -5.0, 0.5, 1.5, 3)
    return Scene("orbit_8x1080p", cams, _mesh(v, f, vcol), g)


def wall4k(seed: int = 4, n_gauss: int = 6_000_000, n_tri: int = 1_000_000) -> Scene:
    """3840x2160; 1M-triangle near-opaque wall; 6M Gaussians, 80% behind it."""
    rng = np.random.default_rng(seed)
    cam = look_at((0, 0, 5), (0, 0, 0), 3840, 2160, 2400, 2400)
    v, f = triangle_soup(rng, n_tri, (-3, -3, 0.9), (3, 3, 1.1), 0.02)
    vcol = rng.uniform(0, 1, size=(len(v), 3))
    n_back = int(round(0.8 * n_gauss))
    back = rng.uniform((-3, -3, -3), (3, 3, 0.5), size=(n_back, 3))
    front = rng.uniform((-3, -3, 1.2), (3, 3, 3), size=(n_gauss - n_back, 3))
    g = _gaussians(rng, np.concatenate([back, front], 0), -5.0, 0.5, 1.5, -1)
    return Scene("wall_4k", [cam], _mesh(v, f, vcol), g)


CONFIGS = {
    "tiny_64": tiny,
    "sphere_512": sphere512,
    "soup_1080p": soup1080,
    "orbit_8x1080p": orbit1080,
    "wall_4k": wall4k,
}


def make(name: str, **kw) -> Scene:
    return CONFIGS[name](**kw)


def upstream_grads(seed: int, width: int, height: int):
    """Seeded dL/d(rgb, depth, alpha) for a loss L = sum(g . out), U[-1, 1]."""
    rng = np.random.default_rng(seed + 1000)
    g_rgb = rng.uniform(-1, 1, size=(height, width, 3)).astype(np.float32)
    g_depth = rng.uniform(-1, 1, size=(height, width)).astype(np.float32)
    g_alpha = rng.uniform(-1, 1, size=(height, width)).astype(np.float32)
    return g_rgb, g_depth, g_alpha


def sample_tiles(seed: int, n_tiles: int, k: int) -> np.ndarray:
    """A seeded sorted sample of ``k`` distinct tile ids (all when k >= n_tiles)."""
    if k >= n_tiles:
        return np.arange(n_tiles, dtype=np.int32)
    rng = np.random.default_rng(seed + 2000)
    return np.sort(rng.choice(n_tiles, size=k, replace=False)).astype(np.int32)


def subset_gaussians(g: Gaussians, idx: np.ndarray) -> Gaussians:
    return Gaussians(g.means[idx], g.log_scales[idx], g.quats[idx], g.logits[idx],
                     g.colors[idx], g.sh_degree)


def empty_mesh() -> Mesh:
    return Mesh(np.zeros((0, 3), np.float32), np.zeros((0, 3), np.int32),
                np.zeros((0, 3), np.float32))


def with_parts(scene: Scene, mesh: Optional[Mesh] = None,
               gaussians: Optional[Gaussians] = None) -> Scene:
    return Scene(scene.name, scene.cameras,
                 scene.mesh if mesh is None else mesh,
                 scene.gaussians if gaussians is None else gaussians, scene.bg)
