"""Seeded synthetic inputs (generators only; no MoE arithmetic lives here)."""
