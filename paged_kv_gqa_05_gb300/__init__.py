"""Placeholder; the binding is added with the library."""
